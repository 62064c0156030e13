// Running (max, sum of exp) pairs and the deterministic mean shared by the
// row kernels and the fused-linear epilogues/finalisers.
//
// The pair (m, s) with s = sum exp(z - m) is the online normaliser of
// Milakov & Gimelshein, "Online normalizer calculation for softmax" (2018):
// two pairs merge into (max, s_a e^{m_a - m} + s_b e^{m_b - m}), so partial
// results over any split of a row combine into the row's log-sum-exp m + ln s.
#pragma once

#include <cmath>
#include <cstdint>

#include "ptx.cuh"

namespace lmho {

struct MS {
  float m;  // running maximum (natural units)
  float s;  // sum of exp(z - m)
};

__device__ __forceinline__ MS ms_empty() { return MS{-INFINITY, 0.f}; }

// Fold n values into (m, s): one rescale per call, one exp per value.
template <int N>
__device__ __forceinline__ void ms_fold(MS& a, const float* v) {
  float vm = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i) vm = fmaxf(vm, v[i]);
  if (vm > a.m) {
    a.s *= ex2_approx((a.m - vm) * kLog2e);
    a.m = vm;
  }
  // all values so far -inf (or masked): exps are 0, NaNs still propagate
  const float nml = (a.m == -INFINITY) ? 0.f : -a.m * kLog2e;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) acc += ex2_approx(fmaf(v[i], kLog2e, nml));
  a.s += acc;
}

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return MS{m, a.s + b.s};
  return MS{m, a.s * ex2_approx((a.m - m) * kLog2e) + b.s * ex2_approx((b.m - m) * kLog2e)};
}

__device__ __forceinline__ MS ms_warp_allreduce(MS a) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    MS b{__shfl_xor_sync(0xFFFFFFFFu, a.m, off), __shfl_xor_sync(0xFFFFFFFFu, a.s, off)};
    a = ms_merge(a, b);
  }
  return a;
}

// Deterministic mean of row_loss[0..T): called by every block that produced
// losses once they are stored; the last of `nwriters` blocks sums them in a
// fixed order in fp64 and writes *loss, then clears the ticket.
__device__ __forceinline__ void mean_tail(const float* row_loss, int64_t T, float* loss, Ctrl* ctrl, uint32_t nwriters) {
  __shared__ uint32_t s_last;
  __shared__ double s_red[32];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&ctrl->ticket, 1u);
    s_last = (prev == nwriters - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nt = blockDim.x;
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < T; i += nt) acc += static_cast<double>(__ldcg(row_loss + i));
  // fixed-order tree: lanes, then warps
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_down_sync(0xFFFFFFFFu, acc, off);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) s_red[w] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int k = 0; k < (nt + 31) / 32; ++k) tot += s_red[k];
    *loss = static_cast<float>(tot / static_cast<double>(T));
    ctrl->ticket = 0u;
    __threadfence();
  }
}

}  // namespace lmho
