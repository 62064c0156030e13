// Row-wise softmax cross-entropy over a [rows, V] logit matrix, fp32 or bf16.
//
// Operation: pages "Cross-entropy loss" (fp32 [tokens, vocab], mean loss[1])
// and "Vocab-parallel cross-entropy, Megatron layout" (bf16 [seq, batch,
// vocab], per-token fp32 loss), section Semantics of each.  For row i:
//   loss_i = m_i + ln(s_i) - z_{i,t_i},  m_i = max_v z_iv,
//   s_i = sum_v exp(z_iv - m_i),
// computed in ONE streaming pass with the online normaliser (Milakov &
// Gimelshein 2018): each thread keeps a running (m, s) and rescales s by
// exp(m_old - m_new) when a new block of values raises the maximum; partial
// (m, s) pairs merge the same way, across lanes, warps and cluster CTAs.
//
// HBM-bound: every logit is read exactly once with 16-byte non-allocating
// loads, several in flight per thread.  Four decompositions of a row:
//   * warp per row   -- small rows; no shared memory, no block barrier;
//   * CTA per row    -- mid/large rows; warp shuffles, then shared memory;
//   * cluster per row -- C CTAs split the row, each merges its share, and CTA 0
//     merges the C partials read from its peers' shared memory (DSMEM);
//   * bulk-copy ring -- rows up to 100 KB whose bytes are 16-byte aligned: one
//     persistent CTA per SM, a producer thread copies whole rows with
//     cp.async.bulk (1-D TMA) into a ring of shared-memory stages (mbarrier
//     complete_tx), and 8 consumer warps each fold whole rows out of shared
//     memory.  Memory-level parallelism is the ring (~200 KB per SM in
//     flight), not registers, so short rows stream at full bandwidth.
// The flat variant's mean is a deterministic two-level sum: per-token losses
// go to the workspace, and the last block to finish (atomic ticket, no spin)
// sums them in a fixed order (compensated fp32, see rowstats.cuh).
#include <cmath>
#include <cstdint>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace lmho {
namespace {

// Partial (m, s) of elements [lo, hi) of one row, shared by `nt` threads
// (this one is `tid`).  Elements before the first 16-byte boundary and after
// the last one are folded one at a time; the aligned body is read as 16-byte
// vectors, U per thread per step, each load instruction coalesced across the
// threads.
template <typename T, int U>
__device__ __forceinline__ MS row_partial(const T* row, int64_t lo, int64_t hi, int tid, int nt) {
  constexpr int E = Elt<T>::kPerVec;
  MS a = ms_empty();
  if (hi <= lo) return a;
  const uintptr_t base = reinterpret_cast<uintptr_t>(row + lo);
  int64_t head = static_cast<int64_t>(((16u - (base & 15u)) & 15u) / sizeof(T));
  if (head > hi - lo) head = hi - lo;
  const int64_t nvec = (hi - lo - head) / E;
  const int64_t body_end = lo + head + nvec * E;
  // scalar head and tail
  for (int64_t j = tid; j < head; j += nt) {
    float v = Elt<T>::load1(row + lo + j);
    ms_fold<1>(a, &v);
  }
  for (int64_t j = body_end + tid; j < hi; j += nt) {
    float v = Elt<T>::load1(row + j);
    ms_fold<1>(a, &v);
  }
  const uint4* vec = reinterpret_cast<const uint4*>(row + lo + head);
  const int64_t step = static_cast<int64_t>(nt) * U;
  constexpr int G = U < 4 ? U : 4;  // vectors per fold (bounds the unpacked registers)
  int64_t q0 = 0;
  // full steps: all U loads in flight, no bounds checks
  for (; q0 + step <= nvec; q0 += step) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ldg_stream_v4(vec + q0 + u * nt + tid);
#pragma unroll
    for (int g = 0; g < U; g += G) {
      float v[G * E];
#pragma unroll
      for (int u = 0; u < G; ++u) Elt<T>::unpack(r[g + u], v + u * E);
      ms_fold<G * E>(a, v);
    }
  }
  // last partial step
  if (q0 < nvec) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t q = q0 + u * nt + tid;
      r[u] = q < nvec ? ldg_stream_v4(vec + q) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int g = 0; g < U; g += G) {
      float v[G * E];
#pragma unroll
      for (int u = 0; u < G; ++u) {
        Elt<T>::unpack(r[g + u], v + u * E);
        if (q0 + (g + u) * nt + tid >= nvec) {
#pragma unroll
          for (int e = 0; e < E; ++e) v[u * E + e] = -INFINITY;
        }
      }
      ms_fold<G * E>(a, v);
    }
  }
  return a;
}

// z[t] of a row, or NaN for a target outside [0, V).  The warp-per-row kernel
// loads t before the row and calls this after it (a load of z[t] that waits
// for t up front would hold back the warp's own row loads); the CTA and
// cluster kernels call it up front from one thread while the others stream.
template <typename T>
__device__ __forceinline__ float target_value(const T* row, int64_t t, int64_t V) {
  return (t >= 0 && t < V) ? Elt<T>::load1(row + t) : __int_as_float(0x7FC00000);
}

__device__ __forceinline__ float finish_loss(MS a, float zt) {
  return a.m + logf(a.s) - zt;
}

// ---------------------------------------------------------------- kernels
// out_rows: per-row losses (per-token output, or the workspace of the flat mean)
// mean_out: non-null for the flat variant.
template <typename T, int U>
__global__ void __launch_bounds__(64) ce_warp_rows(const T* __restrict__ logits,
                                                    const int64_t* __restrict__ target, int64_t rows,
                                                    int64_t V, float* __restrict__ out_rows,
                                                    float* mean_out, Ctrl* ctrl) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r < rows) {
    const T* row = logits + r * V;
    const int64_t t = __ldg(target + r);
    MS a = row_partial<T, U>(row, 0, V, lane, 32);
    a = ms_warp_allreduce(a);
    if (lane == 0)
      out_rows[r] = finish_loss(a, target_value(row, t, V));
  }
  if (mean_out) mean_tail(out_rows, rows, mean_out, ctrl, gridDim.x);
}

template <typename T, int U, int NT>
__global__ void __launch_bounds__(NT) ce_cta_rows(const T* __restrict__ logits,
                                                  const int64_t* __restrict__ target, int64_t rows,
                                                  int64_t V, float* __restrict__ out_rows,
                                                  float* mean_out, Ctrl* ctrl) {
  __shared__ MS s_part[NT / 32];
  const int64_t r = blockIdx.x;
  const T* row = logits + r * V;
  // One thread reads z[t] up front: the CTA's other warps stream meanwhile,
  // and a read at the end would hold the whole CTA (measured 5 % slower for
  // 256 KB bf16 rows).
  float zt = 0.f;
  if (threadIdx.x == 0) zt = target_value(row, __ldg(target + r), V);
  MS a = row_partial<T, U>(row, 0, V, threadIdx.x, NT);
  a = block_allreduce_to0<NT>(a, s_part);
  if (threadIdx.x == 0) out_rows[r] = finish_loss(a, zt);
  if (mean_out) mean_tail(out_rows, rows, mean_out, ctrl, gridDim.x);
}

// Cluster of C CTAs per row; CTA k of the cluster takes the k-th contiguous
// slice of the row (slices cut at 16-byte-vector granularity).
template <typename T, int U, int NT, int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(NT)
    ce_cluster_rows(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t rows,
                    int64_t V, float* __restrict__ out_rows, float* mean_out, Ctrl* ctrl) {
  __shared__ MS s_part[NT / 32];
  __shared__ float s_ms[2];
  const uint32_t rank = cluster_ctarank();
  const int64_t r = blockIdx.x / C;
  const T* row = logits + r * V;
  // slice boundaries in elements, multiples of 64 elements
  const int64_t chunk = ((V + C - 1) / C + 63) / 64 * 64;
  const int64_t lo = (chunk * rank < V) ? chunk * rank : V;
  const int64_t hi = (lo + chunk < V) ? lo + chunk : V;
  float zt = 0.f;  // as in ce_cta_rows
  if (rank == 0 && threadIdx.x == 0) zt = target_value(row, __ldg(target + r), V);
  MS a = row_partial<T, U>(row, lo, hi, threadIdx.x, NT);
  a = block_allreduce_to0<NT>(a, s_part);
  if (threadIdx.x == 0) { s_ms[0] = a.m; s_ms[1] = a.s; }
  cluster_sync();  // partials visible cluster-wide
  if (rank == 0 && threadIdx.x == 0) {
    MS tot{s_ms[0], s_ms[1]};
    for (uint32_t k = 1; k < C; ++k) {
      MS b{ld_dsmem_f32(mapa_shared(&s_ms[0], k)), ld_dsmem_f32(mapa_shared(&s_ms[1], k))};
      tot = ms_merge(tot, b);
    }
    out_rows[r] = finish_loss(tot, zt);
  }
  cluster_sync();  // peers keep their shared memory until CTA 0 has read it
  if (mean_out && rank == 0) mean_tail(out_rows, rows, mean_out, ctrl, gridDim.x / C);
}

// Persistent bulk-copy ring: CTA b takes the contiguous rows [b*per, b*per+n)
// (per = ceil(rows / gridDim.x)), so each SM streams one contiguous range;
// its item i is row b*per + i,
// held in stage i % stages and folded by consumer warp i % nwa, where nwa (the
// active consumer warps) divides `stages`.  So each stage has ONE owner warp,
// which waits on that stage's barrier fill after fill, in order: a parity wait
// is only unambiguous when its waiter is never more than one phase ahead.
// Every wait is bounded; a warp that gives up writes NaN for its remaining
// rows and records the timeout when a status word exists.
template <typename T, int NW>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
    ce_bulk_rows(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t rows, int64_t V,
                 float* __restrict__ out_rows, float* mean_out, Ctrl* ctrl, int stages, int nwa,
                 uint32_t stage_bytes, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(stages) * stage_bytes);
  uint64_t* empty = full + stages;
  uint32_t* status = ctrl ? &ctrl->status : nullptr;
  const uint32_t row_bytes = static_cast<uint32_t>(V * sizeof(T));
  const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t n_items = first < rows ? (rows - first < per ? rows - first : per) : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) {
      uint32_t filled = 0, last_parity = 0;  // stages <= 32
      for (int64_t i = 0; i < n_items; ++i) {
        const int s = static_cast<int>(i % stages);
        const uint32_t k = static_cast<uint32_t>(i / stages);
        if (!mbar_wait(&empty[s], (k & 1u) ^ 1u, timeout_ns, status)) break;
        const int64_t r = first + i;
        mbar_arrive_expect_tx(&full[s], row_bytes);
        bulk_load(ring + static_cast<size_t>(s) * stage_bytes, logits + r * V, row_bytes, &full[s]);
        filled |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | ((k & 1u) << s);
      }
      // never leave with copies in flight
      for (int s = 0; s < stages; ++s)
        if (filled & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, timeout_ns, status);
    }
  } else {
    constexpr int E = Elt<T>::kPerVec;
    const int nvec = static_cast<int>(row_bytes / 16);
    for (int64_t i = warp - 1; warp - 1 < nwa && i < n_items; i += nwa) {
      const int s = static_cast<int>(i % stages);
      const uint32_t k = static_cast<uint32_t>(i / stages);
      const int64_t r = first + i;
      const int64_t t = __ldg(target + r);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], k & 1u, timeout_ns, status))) {
        for (int64_t j = i; j < n_items; j += nwa)
          if (lane == 0) out_rows[first + j] = __int_as_float(0x7FC00000);
        break;
      }
      const uint8_t* row = ring + static_cast<size_t>(s) * stage_bytes;
      const uint4* vec = reinterpret_cast<const uint4*>(row);
      MS a = ms_empty();
      int q = lane;
      for (; q + 96 < nvec; q += 128) {
        uint4 rr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) rr[u] = vec[q + 32 * u];
        float v[4 * E];
#pragma unroll
        for (int u = 0; u < 4; ++u) Elt<T>::unpack(rr[u], v + u * E);
        ms_fold<4 * E>(a, v);
      }
      for (; q < nvec; q += 32) {
        float v[E];
        Elt<T>::unpack(vec[q], v);
        ms_fold<E>(a, v);
      }
      a = ms_warp_allreduce(a);
      if (lane == 0) {
        const float zt = (t >= 0 && t < V) ? Elt<T>::load_any(reinterpret_cast<const T*>(row) + t)
                                           : __int_as_float(0x7FC00000);
        out_rows[r] = finish_loss(a, zt);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  if (mean_out) mean_tail(out_rows, rows, mean_out, ctrl, gridDim.x);
}

template <typename T>
cudaError_t launch_rows(const T* logits, const int64_t* target, int64_t rows, int64_t V,
                        float* out_rows, float* mean_out, Ctrl* ctrl, const CeConfig& cfg,
                        cudaStream_t st) {
  launch_mark(0, st);
  switch (cfg.variant) {
    case kCeWarp: {
      // 16 loads per lane in flight: a 16 KB row takes one or two memory round
      // trips, a 32 KB row four (with 4 in flight, 16; Megatron bf16 V = 16384
      // measured 49.3-49.6 vs 50.1-50.2 us, 64 vs 54 registers).  Blocks of 2
      // warps: Megatron V = 16384 47.6-47.9 us against 49.2 with 8 warps, the
      // same at V = 4096 and 8192, one event tick slower with 16.
      const int64_t blocks = (rows + 1) / 2;
      ce_warp_rows<T, 16><<<static_cast<unsigned>(blocks), 64, 0, st>>>(logits, target, rows, V, out_rows, mean_out,
                                                                         ctrl);
      break;
    }
    case kCeCta:
      if (cfg.threads == 512)
        ce_cta_rows<T, 4, 512><<<static_cast<unsigned>(rows), 512, 0, st>>>(logits, target, rows, V,
                                                                             out_rows, mean_out, ctrl);
      else
        ce_cta_rows<T, 4, 256><<<static_cast<unsigned>(rows), 256, 0, st>>>(logits, target, rows, V,
                                                                             out_rows, mean_out, ctrl);
      break;
    case kCeBulk: {
      const uint32_t row_bytes = static_cast<uint32_t>(V * sizeof(T));
      const uint32_t stage_bytes = (row_bytes + 127) / 128 * 128;
      const uint32_t ring = cfg.bulk_ring_bytes ? cfg.bulk_ring_bytes : kCeBulkRingBytes;
      int stages = static_cast<int>(ring / stage_bytes);
      if (stages > 32) stages = 32;
      // active consumer warps: at least two stages each, so every warp has its
      // next row in flight while it folds the current one
      int nwa = stages / 2;
      nwa = nwa < 1 ? 1 : (nwa > 8 ? 8 : nwa);
      stages = stages / nwa * nwa;               // each stage owned by one warp
      const size_t smem = static_cast<size_t>(stages) * stage_bytes + 128 + 16 * stages;
      static std::atomic<bool> limit_set[kMaxDevices];
      const cudaError_t e =
          ensure_smem_limit(ce_bulk_rows<T, 8>, static_cast<int>(kCeBulkRingBytes + 128 + 16 * 32), limit_set);
      if (e != cudaSuccess) return e;
      int64_t grid = rows < cfg.num_sms ? rows : cfg.num_sms;
      const int64_t per = (rows + grid - 1) / grid;
      grid = (rows + per - 1) / per;   // no CTA without rows
      ce_bulk_rows<T, 8><<<static_cast<unsigned>(grid), 32 * 9, smem, st>>>(logits, target, rows, V, out_rows, mean_out,
                                                                           ctrl, stages, nwa, stage_bytes, cfg.timeout_ns);
      break;
    }
    case kCeCluster: {
      const unsigned grid = static_cast<unsigned>(rows * cfg.cluster);
      if (cfg.cluster == 2)
        ce_cluster_rows<T, 4, 256, 2><<<grid, 256, 0, st>>>(logits, target, rows, V, out_rows, mean_out, ctrl);
      else if (cfg.cluster == 4)
        ce_cluster_rows<T, 4, 256, 4><<<grid, 256, 0, st>>>(logits, target, rows, V, out_rows, mean_out, ctrl);
      else
        ce_cluster_rows<T, 4, 256, 8><<<grid, 256, 0, st>>>(logits, target, rows, V, out_rows, mean_out, ctrl);
      break;
    }
    default:
      return cudaErrorInvalidValue;
  }
  launch_mark(1, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ce_f32(const float* logits, const int64_t* target, int64_t T, int64_t V,
                          float* loss, float* row_loss, Ctrl* ctrl, const CeConfig& cfg,
                          cudaStream_t st) {
  return launch_rows<float>(logits, target, T, V, row_loss, loss, ctrl, cfg, st);
}

cudaError_t launch_ce_bf16_rows(const uint16_t* logits, const int64_t* target, int64_t rows,
                                int64_t V, float* loss_rows, const CeConfig& cfg, cudaStream_t st) {
  return launch_rows<uint16_t>(logits, target, rows, V, loss_rows, nullptr, nullptr, cfg, st);
}

}  // namespace lmho
