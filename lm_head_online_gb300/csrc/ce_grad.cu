// Cross-entropy forward + backward over a [rows, V] logit matrix in one pass
// over HBM: the loss of every row and the gradient with respect to the logits,
//   dz_iv = g_i * (softmax(z_i)_v - [v == t_i]),
// with g_i = grad_scale / T for the flat mean (page "Cross-entropy loss") or
// g_i = grad_scale * dloss_i for per-token losses (page "Vocab-parallel
// cross-entropy, Megatron layout").  The gradient needs the row's
// log-sum-exp before any element can be written, so the logits would be read
// twice; here each row is read once into shared memory and the gradient is
// written from there:
//   * a cluster of C CTAs per row (C = 1 for rows up to 64 KB), CTA k staging
//     the k-th slice (at most 64 KB) while folding the online (max, sum exp).
//     Measured on GB300: one CTA per 64 KB row moves 6.6 TB/s of read + write
//     where a pair of CTAs moved 5.1-5.8; slices of 128 KB or more (one CTA per
//     SM) are slower than clusters of 64 KB slices at every size;
//   * the C slice partials are exchanged through distributed shared memory:
//     each CTA pushes its partial into every peer, one cluster barrier, then
//     every CTA merges them in rank order (all agree bit for bit on the row's
//     log-sum-exp);
//   * each CTA then writes its slice of the gradient, 16-byte stores where the
//     gradient row has the logits' alignment, scalar stores otherwise.
// Aligned rows of at most 16 KB take one or two warps per row instead
// (ce_fb_warp_rows): the row stays in registers between the fold and the
// gradient write.
// When the slice's start and length are multiples of 16 bytes, one thread
// stages it with a single cp.async.bulk (1-D TMA) completing on an mbarrier,
// so the whole slice is in flight at once; otherwise the threads load it
// through registers.  Rows longer than 8 x 64 KB are not staged: the second
// pass re-reads global memory.  A target outside [0, V) makes the row's loss
// and gradient NaN, as does a staging wait that gives up (bounded; recorded
// in the status word when there is one).
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace lmho {
namespace {

constexpr int64_t kSliceMaxBytes = 192 * 1024;   // largest slice a CTA can stage (shared memory)
#ifndef LMHO_FB_WARP
#define LMHO_FB_WARP 1   // one or two warps per row for aligned rows up to 16 KB
#endif

template <typename T> struct Out;
template <> struct Out<float> {
  __device__ static void store1(float* p, float v) { *p = v; }
  __device__ static uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};
template <> struct Out<uint16_t> {
  __device__ static void store1(uint16_t* p, float v) { *p = static_cast<uint16_t>(pack_bf16x2(v, 0.f)); }
  __device__ static uint4 pack(const float* v) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
  }
};

// STAGED: the slice lives in dynamic shared memory between the two passes;
// element j of the row sits at st[pad + (j - lo)], pad chosen so shared and
// global addresses agree modulo 16 bytes.
template <typename T, int C, int NT, bool STAGED>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(NT)
    ce_fb_rows(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t rows, int64_t V,
               int64_t slice, const float* __restrict__ dloss, float gscale, float* __restrict__ out_rows,
               T* __restrict__ dlogits, float* mean_out, Ctrl* ctrl, uint64_t timeout_ns) {
  constexpr int E = Elt<T>::kPerVec;
  constexpr int U = 4;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ MS s_part[NT / 32];
  __shared__ float s_peer[C][2];   // (max, sum exp) of every CTA of the cluster, pushed by its owner
  __shared__ float s_lse;
  __shared__ uint64_t s_bar;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  if (C > 1) cluster_arrive_relaxed();   // barrier phase 0: this CTA is running
  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x / C;
  const T* row = logits + r * V;
  T* drow = dlogits + r * V;
  const int64_t lo = (static_cast<int64_t>(rank) * slice < V) ? static_cast<int64_t>(rank) * slice : V;
  const int64_t hi = (lo + slice < V) ? lo + slice : V;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(row + lo);
  const int pad = static_cast<int>((a0 & 15u) / sizeof(T));
  T* st = reinterpret_cast<T*>(smem_raw) + pad - lo;   // st[j] for j in [lo, hi)
  int64_t head = static_cast<int64_t>(((16u - (a0 & 15u)) & 15u) / sizeof(T));
  if (head > hi - lo) head = hi - lo;
  const int64_t nvec = (hi - lo - head) / E;
  const int64_t body = lo + head, body_end = body + nvec * E;

  // ---- pass 1: read the slice once, fold (max, sum exp), stage it
  MS a = ms_empty();
  const bool tma = STAGED && hi > lo && (a0 & 15u) == 0 && ((hi - lo) * sizeof(T)) % 16 == 0;
  bool ok = true;
  if (tma) {
    if (tid == 0) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, static_cast<uint32_t>((hi - lo) * sizeof(T)));
      bulk_load(st + lo, row + lo, static_cast<uint32_t>((hi - lo) * sizeof(T)), &s_bar);
    }
    __syncthreads();
    ok = __syncthreads_and(mbar_wait(&s_bar, 0, timeout_ns, ctrl ? &ctrl->status : nullptr)) != 0;
    if (ok) {
      const uint4* sv = reinterpret_cast<const uint4*>(st + lo);
      for (int64_t q0 = 0; q0 < nvec; q0 += static_cast<int64_t>(NT) * U) {
        float v[U * E];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t q = q0 + u * NT + tid;
          if (q < nvec) {
            Elt<T>::unpack(sv[q], v + u * E);
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[u * E + e] = -INFINITY;
          }
        }
        ms_fold<U * E>(a, v);
      }
    }
  } else {
    for (int64_t j = lo + tid; j < body; j += NT) {
      float v = Elt<T>::load1(row + j);
      if (STAGED) st[j] = row[j];
      ms_fold<1>(a, &v);
    }
    for (int64_t j = body_end + tid; j < hi; j += NT) {
      float v = Elt<T>::load1(row + j);
      if (STAGED) st[j] = row[j];
      ms_fold<1>(a, &v);
    }
    const uint4* gvec = reinterpret_cast<const uint4*>(row + body);
    uint4* svec = reinterpret_cast<uint4*>(st + body);
    for (int64_t q0 = 0; q0 < nvec; q0 += static_cast<int64_t>(NT) * U) {
      uint4 rr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t q = q0 + u * NT + tid;
        rr[u] = q < nvec ? ldg_stream_v4(gvec + q) : make_uint4(0u, 0u, 0u, 0u);
      }
      float v[U * E];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t q = q0 + u * NT + tid;
        Elt<T>::unpack(rr[u], v + u * E);
        if (q < nvec) {
          if (STAGED) svec[q] = rr[u];
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) v[u * E + e] = -INFINITY;
        }
      }
      ms_fold<U * E>(a, v);
    }
  }
  a = block_allreduce_to0<NT>(a, s_part);

  // ---- the row's log-sum-exp (merged across the cluster in rank order)
  if (C == 1) {
    if (tid == 0) s_lse = a.m + logf(a.s);
  } else {
    // Phase 0 completes at once (every CTA arrived at its start), proving all
    // peers run; each CTA then pushes its partial into every peer's s_peer.
    // After phase 1 every CTA holds all C partials locally and touches no
    // other CTA's shared memory again, so one full barrier suffices.
    cluster_wait();
    if (tid == 0)
      for (uint32_t k = 0; k < C; ++k) {
        st_dsmem_f32(mapa_shared(&s_peer[rank][0], k), a.m);
        st_dsmem_f32(mapa_shared(&s_peer[rank][1], k), a.s);
      }
    cluster_sync();
    if (tid == 0) {
      MS tot = ms_empty();
      for (uint32_t k = 0; k < C; ++k) tot = ms_merge(tot, MS{s_peer[k][0], s_peer[k][1]});
      s_lse = tot.m + logf(tot.s);
    }
  }
  __syncthreads();
  const float lse = s_lse;
  const int64_t t = __ldg(target + r);
  const bool bad = t < 0 || t >= V || !ok;
  const float g = gscale * (dloss ? __ldg(dloss + r) : 1.f);
  const float nl = -lse * kLog2e;

  // ---- pass 2: gradient of the slice.  Every element gets g * softmax; the
  // target element is patched to g * (softmax - 1) after a barrier.
  const T* src = STAGED ? static_cast<const T*>(st) : row;  // st is indexed by row position
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(drow + lo) & 15u) == (a0 & 15u));
  const float nan = __int_as_float(0x7FC00000);
  auto gp = [&](float z) { return bad ? nan : g * ex2_approx(fmaf(z, kLog2e, nl)); };
  if (vec_ok) {
    for (int64_t j = lo + tid; j < body; j += NT) Out<T>::store1(drow + j, gp(Elt<T>::load_any(src + j)));
    for (int64_t j = body_end + tid; j < hi; j += NT) Out<T>::store1(drow + j, gp(Elt<T>::load_any(src + j)));
    const uint4* sv = reinterpret_cast<const uint4*>(src + body);
    uint4* dv = reinterpret_cast<uint4*>(drow + body);
    if (bad) {
      float o[E];
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = nan;
      const uint4 w = Out<T>::pack(o);
      for (int64_t q = tid; q < nvec; q += NT) dv[q] = w;
    } else {
      for (int64_t q = tid; q < nvec; q += NT) {
        const uint4 raw = STAGED ? sv[q] : ldg_stream_v4(sv + q);
        float v[E];
        Elt<T>::unpack(raw, v);
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = g * ex2_approx(fmaf(v[e], kLog2e, nl));
        dv[q] = Out<T>::pack(v);
      }
    }
  } else {
    for (int64_t j = lo + tid; j < hi; j += NT) Out<T>::store1(drow + j, gp(Elt<T>::load_any(src + j)));
  }
  if (!bad && t >= lo && t < hi) {
    __syncthreads();  // the patch lands after the bulk store of the same element
    if (tid == 0) Out<T>::store1(drow + t, g * (ex2_approx(fmaf(Elt<T>::load_any(src + t), kLog2e, nl)) - 1.f));
  }

  // ---- the row's loss
  if (rank == 0 && tid == 0) {
    const float zt = (t < 0 || t >= V) ? __int_as_float(0x7FC00000) : Elt<T>::load1(row + t);
    out_rows[r] = ok ? lse - zt : __int_as_float(0x7FC00000);
  }
  if (mean_out && rank == 0) mean_tail(out_rows, rows, mean_out, ctrl, gridDim.x / C);
}

// Rows of at most W x 32 x U 16-byte vectors, 16-byte aligned and whole
// vectors (logits and gradient): W warps per row (W = 1: two rows per 64-thread
// block; W = 2: one) hold the row in registers, U vectors per lane
// lane-interleaved as in the forward warp kernel, fold (max, sum exp), merge
// across the warp and then, for W = 2, through shared memory in warp order, so
// both warps hold the same log-sum-exp.  The gradient is written from the same
// registers; thread 0 of the row then patches the target element (after a
// barrier, so it lands after the vector store covering it) and writes the
// row's loss.  One read of the logits and one write of the gradient, with no
// shared-memory staging of the row.  The flat mean is a one-block kernel
// launched behind this one as a programmatic dependent.
template <typename T, int U, int G, int W>
__global__ void __launch_bounds__(64) ce_fb_warp_rows(const T* __restrict__ logits, const int64_t* __restrict__ target,
                                                     int64_t rows, int64_t V, const float* __restrict__ dloss,
                                                     float gscale, float* __restrict__ out_rows,
                                                     T* __restrict__ dlogits) {
  static_assert(W == 1 || W == 2, "one or two warps per row");
  constexpr int E = Elt<T>::kPerVec;
  __shared__ float s_ms[2][2];
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t r = W == 1 ? static_cast<int64_t>(blockIdx.x) * 2 + w : static_cast<int64_t>(blockIdx.x);
  const int64_t q_lo = W == 1 ? 0 : static_cast<int64_t>(w) * 32 * U;   // this warp's first vector
  const bool live = r < rows;
  const T* row = logits + (live ? r : 0) * V;
  const int64_t nvec = V / E;
  const uint4* vec = reinterpret_cast<const uint4*>(row);
  uint4 rv[U];
  MS a = ms_empty();
  int64_t t = 0;
  if (live) {
    t = __ldg(target + r);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t q = q_lo + u * 32 + lane;
      rv[u] = q < nvec ? ldg_stream_v4(vec + q) : neg_inf_vec<T>();
    }
#pragma unroll
    for (int gi = 0; gi < U; gi += G) ms_fold_vecs<T, G>(a, rv + gi);
    a = ms_warp_allreduce(a);
  }
  if constexpr (W == 2) {
    if (lane == 0) {
      s_ms[w][0] = a.m;
      s_ms[w][1] = a.s;
    }
    __syncthreads();
    a = ms_merge(MS{s_ms[0][0], s_ms[0][1]}, MS{s_ms[1][0], s_ms[1][1]});
  }
  const float lse = a.m + logf(a.s);
  const bool bad = t < 0 || t >= V;
  const float g = live ? gscale * (dloss ? __ldg(dloss + r) : 1.f) : 0.f;
  const float nl = -lse * kLog2e;
  const float nan = __int_as_float(0x7FC00000);
  if (live) {
    uint4* dv = reinterpret_cast<uint4*>(dlogits + r * V);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t q = q_lo + u * 32 + lane;
      if (q < nvec) {
        float v[E];
        Elt<T>::unpack(rv[u], v);
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = bad ? nan : g * ex2_approx(fmaf(v[e], kLog2e, nl));
        dv[q] = Out<T>::pack(v);
      }
    }
  }
  if constexpr (W == 2)
    __syncthreads();
  else
    __syncwarp();
  if (live && lane == 0 && (W == 1 || w == 0)) {
    const float zt = bad ? nan : Elt<T>::load1(row + t);
    if (!bad) Out<T>::store1(dlogits + r * V + t, g * (ex2_approx(fmaf(zt, kLog2e, nl)) - 1.f));
    out_rows[r] = lse - zt;
  }
}

// Mean of the row losses behind ce_fb_warp_rows (a programmatic dependent:
// griddep_wait returns once that grid has completed and its writes are visible).
__global__ void __launch_bounds__(256) fb_mean_rows(const float* __restrict__ out_rows, int64_t rows, float* loss) {
  griddep_wait();
  mean_sum(out_rows, rows, loss);
}

template <typename T, int U, int G, int W>
cudaError_t launch_fb_warp(const T* logits, const int64_t* target, int64_t rows, int64_t V, const float* dloss,
                           float gscale, float* out_rows, T* dlogits, float* mean_out, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>(W == 1 ? (rows + 1) / 2 : rows);
  ce_fb_warp_rows<T, U, G, W><<<blocks, 64, 0, st>>>(logits, target, rows, V, dloss, gscale, out_rows, dlogits);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  if (!mean_out) return cudaSuccess;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(1);
  lc.blockDim = dim3(256);
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fb_mean_rows, static_cast<const float*>(out_rows), rows, mean_out);
}

template <typename T, int C, int NT, bool STAGED>
cudaError_t launch_fb(const T* logits, const int64_t* target, int64_t rows, int64_t V, int64_t slice,
                      const float* dloss, float gscale, float* out_rows, T* dlogits, float* mean_out, Ctrl* ctrl,
                      uint64_t timeout_ns, cudaStream_t st) {
  const size_t smem = STAGED ? static_cast<size_t>(slice) * sizeof(T) + 16 : 0;
  auto kern = ce_fb_rows<T, C, NT, STAGED>;
  if (smem > 48 * 1024) {
    static std::atomic<bool> limit_set[kMaxDevices];
    const cudaError_t e = ensure_smem_limit(kern, static_cast<int>(kSliceMaxBytes + 16), limit_set);
    if (e != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(rows * C), NT, smem, st>>>(logits, target, rows, V, slice, dloss, gscale, out_rows,
                                                          dlogits, mean_out, ctrl, timeout_ns);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fb_rows(const T* logits, const int64_t* target, int64_t rows, int64_t V, const float* dloss,
                           float gscale, float* out_rows, T* dlogits, float* mean_out, Ctrl* ctrl, uint64_t tmo,
                           cudaStream_t st) {
  const int64_t row_bytes = V * static_cast<int64_t>(sizeof(T));
  auto slice_for = [&](int c) {  // elements per CTA, a multiple of 64
    return ((V + c - 1) / c + 63) / 64 * 64;
  };
  // Largest slice a cluster CTA stages (default 64 KB) and longest row one CTA
  // stages alone (default 64 KB); LMHO_FB_SLICE_KB / LMHO_FB_SINGLE_KB = 16..192
  // override them for sweeps.
  auto knob = [](const char* name, int64_t dflt) {
    const char* v = std::getenv(name);
    const long kb = v ? std::strtol(v, nullptr, 10) : 0;
    return (kb >= 16 && kb * 1024 <= kSliceMaxBytes) ? static_cast<int64_t>(kb) * 1024 : dflt;
  };
  static const int64_t cap = knob("LMHO_FB_SLICE_KB", 64 * 1024);
  static const int64_t single = knob("LMHO_FB_SINGLE_KB", 64 * 1024);
  launch_mark(0, st);
  cudaError_t e;
  // warp per row for short aligned rows (logits and gradient rows on 16-byte boundaries)
  constexpr int G = sizeof(T) == 2 ? 16 : 4;   // vectors per fold, as in the forward warp kernel
  const bool rows_aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 &&
                            (reinterpret_cast<uintptr_t>(dlogits) & 15u) == 0 && row_bytes % 16 == 0;
  // Rows up to 8 KB: one warp per row; up to 16 KB: two.  Measured on GB300
  // (flushed calls, against the staged CTA kernel): bf16 [2048 x 4, V] 35.1 ->
  // 23.7-24.0 us at V = 4096 and 49.5 -> 43.0 us at 8192; fp32 [16384, V]
  // 78.1-78.5 -> 45.8-46.2 us at V = 2048 and 104.2 -> 83.5 us at 4096.  One
  // warp holding a whole 16 KB row (32 vectors per lane) spills or runs slower.
  if (LMHO_FB_WARP && rows_aligned && row_bytes <= 32 * 16 * 16)
    e = launch_fb_warp<T, 16, G, 1>(logits, target, rows, V, dloss, gscale, out_rows, dlogits, mean_out, st);
  else if (LMHO_FB_WARP && rows_aligned && row_bytes <= 2 * 32 * 16 * 16)
    e = launch_fb_warp<T, 16, G, 2>(logits, target, rows, V, dloss, gscale, out_rows, dlogits, mean_out, st);
  else if (row_bytes <= 16 * 1024)
    e = launch_fb<T, 1, 128, true>(logits, target, rows, V, slice_for(1), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  else if (row_bytes <= single)
    e = launch_fb<T, 1, 256, true>(logits, target, rows, V, slice_for(1), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  // fp32 rows over 96 KB and up to 128 KB: four CTAs of 24-32 KB slices.  At 128
  // KB (V = 32768) they took 673-674 us against two 64 KB slices' 721-723 us
  // (T = 16384) and 176 vs 190-191 us (T = 4096); bf16 rows of that size, and
  // 256 KB rows of either type, were slower with the smaller slices.
  else if (sizeof(T) == 4 && row_bytes > 96 * 1024 && row_bytes <= 128 * 1024 && cap == 64 * 1024)
    e = launch_fb<T, 4, 256, true>(logits, target, rows, V, slice_for(4), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  else if (slice_for(2) * static_cast<int64_t>(sizeof(T)) <= cap)
    e = launch_fb<T, 2, 256, true>(logits, target, rows, V, slice_for(2), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  else if (slice_for(4) * static_cast<int64_t>(sizeof(T)) <= cap)
    e = launch_fb<T, 4, 256, true>(logits, target, rows, V, slice_for(4), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  else if (slice_for(8) * static_cast<int64_t>(sizeof(T)) <= cap)
    e = launch_fb<T, 8, 256, true>(logits, target, rows, V, slice_for(8), dloss, gscale, out_rows, dlogits, mean_out,
                                   ctrl, tmo, st);
  else
    e = launch_fb<T, 8, 256, false>(logits, target, rows, V, slice_for(8), dloss, gscale, out_rows, dlogits,
                                    mean_out, ctrl, tmo, st);
  launch_mark(1, st);
  return e;
}

}  // namespace

cudaError_t launch_ce_fwd_bwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V, float gscale,
                                  float* loss, float* row_loss, float* dlogits, Ctrl* ctrl, uint64_t timeout_ns,
                                  cudaStream_t st) {
  return launch_fb_rows<float>(logits, target, T, V, nullptr, gscale, row_loss, dlogits, loss, ctrl, timeout_ns, st);
}

cudaError_t launch_ce_fwd_bwd_bf16_rows(const uint16_t* logits, const int64_t* target, int64_t rows, int64_t V,
                                        const float* dloss, float gscale, float* loss_rows, uint16_t* dlogits,
                                        uint64_t timeout_ns, cudaStream_t st) {
  return launch_fb_rows<uint16_t>(logits, target, rows, V, dloss, gscale, loss_rows, dlogits, nullptr, nullptr,
                                  timeout_ns, st);
}

}  // namespace lmho
