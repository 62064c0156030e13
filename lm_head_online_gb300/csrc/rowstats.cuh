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

// ---------------------------------------------------------------- element types
template <typename T> struct Elt;
template <> struct Elt<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static float load1(const float* p) { return __ldg(p); }
  __device__ static float load_any(const float* p) { return *p; }
  __device__ static void unpack(const uint4& r, float* v) {
    v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
    v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
  }
};
template <> struct Elt<uint16_t> {  // bf16 bit patterns
  static constexpr int kPerVec = 8;
  __device__ static float load1(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
  __device__ static float load_any(const uint16_t* p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }
  __device__ static void unpack(const uint4& r, float* v) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
};

// ---------------------------------------------------------------- packed folds
// Packed fp32 pairs (sm_100+): one instruction does two fp32 FMAs or adds.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f32x2_split(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// max of three fp32 values in one instruction (sm_100+)
__device__ __forceinline__ float max3_f32(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// A 16-byte vector of -inf in the element type (the fill of masked lanes).
template <typename T> __device__ __forceinline__ uint4 neg_inf_vec();
template <> __device__ __forceinline__ uint4 neg_inf_vec<float>() {
  return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}
template <> __device__ __forceinline__ uint4 neg_inf_vec<uint16_t>() {
  return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}

// Maximum of the elements of N raw 16-byte vectors (NaNs are dropped here;
// they still reach the sum below and make it NaN).
template <typename T, int N> __device__ __forceinline__ float vec_max(const uint4* r);
template <int N> struct VecMaxF32 {
  static __device__ __forceinline__ float run(const uint4* r) {
    float m = max3_f32(__uint_as_float(r[0].x), __uint_as_float(r[0].y), __uint_as_float(r[0].z));
    m = fmaxf(m, __uint_as_float(r[0].w));
#pragma unroll
    for (int i = 1; i < N; ++i) {
      m = max3_f32(m, __uint_as_float(r[i].x), __uint_as_float(r[i].y));
      m = max3_f32(m, __uint_as_float(r[i].z), __uint_as_float(r[i].w));
    }
    return m;
  }
};
template <> __device__ __forceinline__ float vec_max<float, 1>(const uint4* r) { return VecMaxF32<1>::run(r); }
template <> __device__ __forceinline__ float vec_max<float, 2>(const uint4* r) { return VecMaxF32<2>::run(r); }
template <> __device__ __forceinline__ float vec_max<float, 4>(const uint4* r) { return VecMaxF32<4>::run(r); }
template <> __device__ __forceinline__ float vec_max<float, 16>(const uint4* r) { return VecMaxF32<16>::run(r); }
template <int N> struct VecMaxBf16 {
  // on the packed words: max.bf16x2 compares two elements per instruction
  static __device__ __forceinline__ float run(const uint4* r) {
    uint32_t w = max_bf16x2(max_bf16x2(r[0].x, r[0].y), max_bf16x2(r[0].z, r[0].w));
#pragma unroll
    for (int i = 1; i < N; ++i) w = max_bf16x2(w, max_bf16x2(max_bf16x2(r[i].x, r[i].y), max_bf16x2(r[i].z, r[i].w)));
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
};
template <> __device__ __forceinline__ float vec_max<uint16_t, 1>(const uint4* r) { return VecMaxBf16<1>::run(r); }
template <> __device__ __forceinline__ float vec_max<uint16_t, 2>(const uint4* r) { return VecMaxBf16<2>::run(r); }
template <> __device__ __forceinline__ float vec_max<uint16_t, 4>(const uint4* r) { return VecMaxBf16<4>::run(r); }
template <> __device__ __forceinline__ float vec_max<uint16_t, 16>(const uint4* r) { return VecMaxBf16<16>::run(r); }

// Fold N raw 16-byte vectors into (m, s): the max first (one rescale of s
// when it rises), then exp(z - m) of every element with the exponent
// argument z log2e - m log2e formed two elements per FMA and the terms summed
// two per add.  Same arithmetic as ms_fold (fp32 FMA, ex2.approx, fp32 sums);
// about half the instructions per element.
template <typename T, int N>
__device__ __forceinline__ void ms_fold_vecs(MS& a, const uint4* r) {
  const float vm = vec_max<T, N>(r);
  if (vm > a.m) {
    a.s *= ex2_approx((a.m - vm) * kLog2e);
    a.m = vm;
  }
  const float nml = (a.m == -INFINITY) ? 0.f : -a.m * kLog2e;  // all -inf so far: terms are 0
  const uint64_t l2e = f32x2(kLog2e, kLog2e), off = f32x2(nml, nml);
  uint64_t acc = f32x2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
    if constexpr (sizeof(T) == 4) {
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        float e0, e1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(w[k]), __uint_as_float(w[k + 1])), l2e, off), e0, e1);
        acc = add_f32x2(acc, f32x2(ex2_approx(e0), ex2_approx(e1)));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float e0, e1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u)), l2e, off),
                    e0, e1);
        acc = add_f32x2(acc, f32x2(ex2_approx(e0), ex2_approx(e1)));
      }
    }
  }
  float s0, s1;
  f32x2_split(acc, s0, s1);
  a.s += s0 + s1;
}

// ms_fold over N fp32 values (N a multiple of 4) with the same steps as
// ms_fold_vecs: a 3-input max, one rescale of s when it rises, and the
// exponent arguments and the sum two values per fp32x2 instruction.
template <int N>
__device__ __forceinline__ void ms_fold_packed(MS& a, const float* v) {
  static_assert(N % 4 == 0, "pairs of pairs");
  float vm = max3_f32(v[0], v[1], v[2]);
#pragma unroll
  for (int i = 3; i + 1 < N; i += 2) vm = max3_f32(vm, v[i], v[i + 1]);
  vm = fmaxf(vm, v[N - 1]);
  if (vm > a.m) {
    a.s *= ex2_approx((a.m - vm) * kLog2e);
    a.m = vm;
  }
  const float nml = (a.m == -INFINITY) ? 0.f : -a.m * kLog2e;
  const uint64_t l2e = f32x2(kLog2e, kLog2e), off = f32x2(nml, nml);
  uint64_t acc = f32x2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    float e0, e1;
    f32x2_split(fma_f32x2(f32x2(v[i], v[i + 1]), l2e, off), e0, e1);
    acc = add_f32x2(acc, f32x2(ex2_approx(e0), ex2_approx(e1)));
  }
  float s0, s1;
  f32x2_split(acc, s0, s1);
  a.s += s0 + s1;
}

template <int NT>
__device__ __forceinline__ MS block_allreduce_to0(MS a, MS* s_part) {
  a = ms_warp_allreduce(a);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) s_part[w] = a;
  __syncthreads();
  MS tot = s_part[0];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 1; k < NT / 32; ++k) tot = ms_merge(tot, s_part[k]);
  }
  return tot;  // valid in thread 0
}

// Compensated (Kahan) fp32 sum: ~1 ulp of the total regardless of the number
// of terms, without fp64 arithmetic (whose rate on this part is a small
// fraction of fp32).
struct KSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// Deterministic mean of row_loss[0..T) (16-byte aligned), computed by the
// whole calling block and written to *loss by thread 0.  The summation order
// is fixed and independent of the block size: 256 virtual lanes each take
// every 256th float4 in index order (compensated fp32, 16 or 8 loads in
// flight); warp 0 then folds 8 lane sums per lane (compensated) and finishes
// with a butterfly whose partners add the same two values.  No fp64: its rate
// on this part is a small fraction of fp32 and a serial fp64 tail costs tens
// of microseconds.  With a keep mask (uint8 per row, may be null) left-out
// rows count as 0 whatever row_loss holds there, and the divisor is the number
// of kept rows (a mean over no row is 0).  Loads bypass L1 (the rows were
// written by other blocks or another grid).
__device__ __forceinline__ float4 keep_only(float4 q, const uint8_t* keep, int64_t r0) {
  if (!__ldg(keep + r0)) q.x = 0.f;
  if (!__ldg(keep + r0 + 1)) q.y = 0.f;
  if (!__ldg(keep + r0 + 2)) q.z = 0.f;
  if (!__ldg(keep + r0 + 3)) q.w = 0.f;
  return q;
}
__device__ __forceinline__ void mean_sum(const float* row_loss, int64_t T, float* loss, const uint8_t* keep = nullptr,
                                         float* inv_count_out = nullptr) {
  constexpr int kVL = 256;
  __shared__ float s_part[kVL];
  __shared__ int64_t s_cnt[kVL];
  const int64_t n4 = T / 4;
  const float4* v4 = reinterpret_cast<const float4*>(row_loss);
  for (int j = threadIdx.x; j < kVL; j += blockDim.x) {
    KSum a;
    int64_t cnt = 0;
    if (keep)
      for (int64_t r = j; r < T; r += kVL) cnt += __ldg(keep + r) != 0;
    s_cnt[j] = cnt;
    int64_t i = j;
    for (; i + 15 * kVL < n4; i += 16 * kVL) {  // 16 loads in flight (T = 16384: one round trip)
      float4 q[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = __ldcg(v4 + i + k * kVL);
      if (keep) {
#pragma unroll
        for (int k = 0; k < 16; ++k) q[k] = keep_only(q[k], keep, 4 * (i + k * kVL));
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        a.add(q[k].x); a.add(q[k].y); a.add(q[k].z); a.add(q[k].w);
      }
    }
    for (; i + 7 * kVL < n4; i += 8 * kVL) {
      float4 q[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) q[k] = __ldcg(v4 + i + k * kVL);
      if (keep) {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = keep_only(q[k], keep, 4 * (i + k * kVL));
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        a.add(q[k].x); a.add(q[k].y); a.add(q[k].z); a.add(q[k].w);
      }
    }
    for (; i < n4; i += kVL) {
      float4 q = __ldcg(v4 + i);
      if (keep) q = keep_only(q, keep, 4 * i);
      a.add(q.x); a.add(q.y); a.add(q.z); a.add(q.w);
    }
    if (j == 0)
      for (int64_t r = n4 * 4; r < T; ++r) a.add((keep && !__ldg(keep + r)) ? 0.f : __ldcg(row_loss + r));
    s_part[j] = a.s - a.c;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    KSum a;
    int64_t n = 0;
#pragma unroll
    for (int k = 0; k < kVL / 32; ++k) {
      a.add(s_part[threadIdx.x * (kVL / 32) + k]);
      n += s_cnt[threadIdx.x * (kVL / 32) + k];
    }
    float v = a.s - a.c;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      n += __shfl_xor_sync(0xFFFFFFFFu, n, off);
    }
    if (threadIdx.x == 0) {
      const int64_t count = keep ? n : T;
      *loss = count > 0 ? v / static_cast<float>(count) : 0.f;
      if (inv_count_out) *inv_count_out = count > 0 ? 1.f / static_cast<float>(count) : 0.f;
    }
  }
}

// The same mean, taken inside a grid whose `nwriters` blocks each produced
// some of the rows: called by every such block once its rows are stored; the
// last block to arrive (atomic ticket, no spin) computes the mean and clears
// the ticket.
__device__ __forceinline__ void mean_tail(const float* row_loss, int64_t T, float* loss, Ctrl* ctrl, uint32_t nwriters,
                                          const uint8_t* keep = nullptr, float* inv_count_out = nullptr) {
  __shared__ uint32_t s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&ctrl->ticket, 1u);
    s_last = (prev == nwriters - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  mean_sum(row_loss, T, loss, keep, inv_count_out);
  if (threadIdx.x == 0) {
    ctrl->ticket = 0u;
    __threadfence();
  }
}

}  // namespace lmho
