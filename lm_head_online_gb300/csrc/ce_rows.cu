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
// The flat variant's mean is a deterministic two-level sum: the row kernel
// writes per-token losses to the workspace, and a one-block kernel launched
// behind it as a programmatic dependent (it is scheduled while the row kernel
// drains, and waits for that grid's completion) sums them in a fixed order
// (compensated fp32, see rowstats.cuh).  The row kernels themselves keep no
// ticket: a fence and an atomic before every block's exit lengthened each
// block's life and held back the next wave (fp32 [16384, 4096] with 8192
// two-warp blocks: 53 us with the in-kernel ticket, 46 us this way).
#include <cmath>
#include <cstdint>
#include <utility>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

// Row kernels launched as programmatic dependents (1, the default) or plainly (0).
#ifndef LMHO_CE_PDL
#define LMHO_CE_PDL 1
#endif
#ifndef LMHO_CE_F32_FOLD
#define LMHO_CE_F32_FOLD 4   // fp32 vectors per fold of the warp-per-row kernel
#endif

namespace lmho {
namespace {

// Partial (m, s) of elements [lo, hi) of one row, shared by `nt` threads
// (this one is `tid`).  Elements before the first 16-byte boundary and after
// the last one are folded one at a time; the aligned body is read as 16-byte
// vectors, U per thread per step, each load instruction coalesced across the
// threads, and folded G vectors at a time (ms_fold_vecs: packed max, packed
// fp32 pairs).  ALIGNED: the caller guarantees row + lo is 16-byte aligned and
// (hi - lo) a whole number of vectors, so there is no scalar head or tail (and
// no registers held for one).
template <typename T, int U, int G, bool ALIGNED = false>
__device__ __forceinline__ MS row_partial(const T* row, int64_t lo, int64_t hi, int tid, int nt) {
  constexpr int E = Elt<T>::kPerVec;
  MS a = ms_empty();
  if (hi <= lo) return a;
  int64_t head = 0, nvec = (hi - lo) / E;
  if constexpr (!ALIGNED) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(row + lo);
    head = static_cast<int64_t>(((16u - (base & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    nvec = (hi - lo - head) / E;
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
  }
  const uint4* vec = reinterpret_cast<const uint4*>(row + lo + head);
  const int64_t step = static_cast<int64_t>(nt) * U;
  int64_t q0 = 0;
  // full steps: all U loads in flight, no bounds checks, folded in groups of G
  for (; q0 + step <= nvec; q0 += step) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ldg_stream_v4(vec + q0 + u * nt + tid);
#pragma unroll
    for (int g = 0; g < U; g += G) ms_fold_vecs<T, G>(a, r + g);
  }
  // last partial step: vectors past the end read as -inf
  if (q0 < nvec) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t q = q0 + u * nt + tid;
      r[u] = q < nvec ? ldg_stream_v4(vec + q) : neg_inf_vec<T>();
    }
#pragma unroll
    for (int g = 0; g < U; g += G) ms_fold_vecs<T, G>(a, r + g);
  }
  return a;
}

// Where a row's result goes.
//  * LossSink: the row's loss m + ln s - z_t; a target outside [0, V) gives NaN.
//  * PartialSink: one vocabulary shard's partial of the row (vocab-parallel
//    cross-entropy: the row holds the global columns [v0, v0 + V)): its max m,
//    its sum of exp(z - m) s, and the target logit, or -inf when the (global)
//    target is not in this shard; three arrays of `rows` floats.
struct LossSink {
  float* out;
  __device__ __forceinline__ int64_t local(int64_t t, int64_t V) const { return (t >= 0 && t < V) ? t : -1; }
  __device__ __forceinline__ float missing() const { return __int_as_float(0x7FC00000); }
  __device__ __forceinline__ void put(int64_t r, MS a, float zt) const { out[r] = a.m + logf(a.s) - zt; }
  __device__ __forceinline__ void fail(int64_t r) const { out[r] = __int_as_float(0x7FC00000); }
};
struct PartialSink {
  float* m;
  float* s;
  float* z;
  int64_t v0;
  __device__ __forceinline__ int64_t local(int64_t t, int64_t V) const {
    return (t >= v0 && t - v0 < V) ? t - v0 : -1;
  }
  __device__ __forceinline__ float missing() const { return -INFINITY; }
  __device__ __forceinline__ void put(int64_t r, MS a, float zt) const {
    m[r] = a.m;
    s[r] = a.s;
    z[r] = zt;
  }
  __device__ __forceinline__ void fail(int64_t r) const {
    m[r] = s[r] = z[r] = __int_as_float(0x7FC00000);
  }
};

// z[t] of a row for the sink (NaN or -inf when the target is not the row's).
// The warp-per-row kernel loads t before the row and calls this after it (a
// load of z[t] that waits for t up front would hold back the warp's own row
// loads); the CTA and cluster kernels call it up front from one thread while
// the others stream.
template <typename T, class Sink>
__device__ __forceinline__ float target_value(const T* row, int64_t t, int64_t V, const Sink& k) {
  const int64_t l = k.local(t, V);
  return l >= 0 ? Elt<T>::load1(row + l) : k.missing();
}

// ---------------------------------------------------------------- kernels
// sink: where each row's result goes (per-row losses, or a shard's partials).
// Every row kernel lets a programmatic dependent (the flat mean) launch at once.
// Warp per row, U loads per lane in flight, folded G vectors at a time;
// MINB = resident 2-warp blocks per SM the register allocation must allow;
// ALIGNED = every row starts on a 16-byte boundary and is whole vectors long.
template <typename T, int U, int G, int MINB, bool ALIGNED, class Sink>
__global__ void __launch_bounds__(64, MINB) ce_warp_rows(const T* __restrict__ logits,
                                                    const int64_t* __restrict__ target, int64_t rows,
                                                    int64_t V, Sink sink) {
  griddep_launch_dependents();
#if LMHO_CE_PDL
  griddep_wait();  // a programmatic launch: the preceding grid's writes are visible from here
#endif
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r < rows) {
    const T* row = logits + r * V;
    const int64_t t = __ldg(target + r);
    MS a = row_partial<T, U, G, ALIGNED>(row, 0, V, lane, 32);
    a = ms_warp_allreduce(a);
    if (lane == 0) sink.put(r, a, target_value(row, t, V, sink));
  }
}

template <typename T, int U, int NT, class Sink>
__global__ void __launch_bounds__(NT) ce_cta_rows(const T* __restrict__ logits,
                                                  const int64_t* __restrict__ target, int64_t rows,
                                                  int64_t V, Sink sink) {
  griddep_launch_dependents();
#if LMHO_CE_PDL
  griddep_wait();  // a programmatic launch: the preceding grid's writes are visible from here
#endif
  __shared__ MS s_part[NT / 32];
  const int64_t r = blockIdx.x;
  const T* row = logits + r * V;
  // One thread reads z[t] up front: the CTA's other warps stream meanwhile,
  // and a read at the end would hold the whole CTA (measured 5 % slower for
  // 256 KB bf16 rows).
  float zt = 0.f;
  if (threadIdx.x == 0) zt = target_value(row, __ldg(target + r), V, sink);
  MS a = row_partial<T, U, U>(row, 0, V, threadIdx.x, NT);
  a = block_allreduce_to0<NT>(a, s_part);
  if (threadIdx.x == 0) sink.put(r, a, zt);
}

// Cluster of C CTAs per row; CTA k of the cluster takes the k-th contiguous
// slice of the row (slices cut at 16-byte-vector granularity).
template <typename T, int U, int NT, int C, class Sink>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(NT)
    ce_cluster_rows(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t rows,
                    int64_t V, Sink sink) {
  griddep_launch_dependents();
#if LMHO_CE_PDL
  griddep_wait();  // a programmatic launch: the preceding grid's writes are visible from here
#endif
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
  if (rank == 0 && threadIdx.x == 0) zt = target_value(row, __ldg(target + r), V, sink);
  MS a = row_partial<T, U, U>(row, lo, hi, threadIdx.x, NT);
  a = block_allreduce_to0<NT>(a, s_part);
  if (threadIdx.x == 0) { s_ms[0] = a.m; s_ms[1] = a.s; }
  cluster_sync();  // partials visible cluster-wide
  if (rank == 0 && threadIdx.x == 0) {
    MS tot{s_ms[0], s_ms[1]};
    for (uint32_t k = 1; k < C; ++k) {
      MS b{ld_dsmem_f32(mapa_shared(&s_ms[0], k)), ld_dsmem_f32(mapa_shared(&s_ms[1], k))};
      tot = ms_merge(tot, b);
    }
    sink.put(r, tot, zt);
  }
  cluster_sync();  // peers keep their shared memory until CTA 0 has read it
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
template <typename T, int NW, class Sink>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
    ce_bulk_rows(const T* __restrict__ logits, const int64_t* __restrict__ target, int64_t rows, int64_t V,
                 Sink sink, Ctrl* ctrl, int stages, int nwa,
                 uint32_t stage_bytes, uint64_t timeout_ns) {
  griddep_launch_dependents();
#if LMHO_CE_PDL
  griddep_wait();  // a programmatic launch: the preceding grid's writes are visible from here
#endif
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
          if (lane == 0) sink.fail(first + j);
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
        const int64_t l = sink.local(t, V);
        const float zt = l >= 0 ? Elt<T>::load_any(reinterpret_cast<const T*>(row) + l) : sink.missing();
        sink.put(r, a, zt);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// Mean of the per-row losses, one block of 256 threads, launched behind the
// row kernel as a programmatic dependent: griddep_wait() returns once that
// grid has completed and its row losses are visible.
__global__ void __launch_bounds__(256) ce_mean_rows(const float* __restrict__ out_rows, int64_t rows,
                                                     float* mean_out) {
  griddep_wait();
  mean_sum(out_rows, rows, mean_out);
}

// Vocab-parallel cross-entropy: the loss of each row from `shards` shards'
// partials (shard j's m, s and z at part + (3 j + {0, 1, 2}) rows), merged in
// shard order: (M, S) by the online-normaliser merge, the target logit as the
// largest of the shards' values (all but the owning shard hold -inf; a NaN
// propagates).  A target outside [0, V) gives NaN.
__global__ void __launch_bounds__(256) ce_merge_rows(const float* __restrict__ part, int64_t shards,
                                                      const int64_t* __restrict__ target, int64_t rows,
                                                      int64_t V, float* __restrict__ loss) {
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = __ldg(target + r);
    MS tot = ms_empty();
    float z = -INFINITY;
    for (int64_t j = 0; j < shards; ++j) {
      const float* p = part + 3 * j * rows;
      tot = ms_merge(tot, MS{__ldg(p + r), __ldg(p + rows + r)});
      const float zj = __ldg(p + 2 * rows + r);
      if (zj > z || zj != zj) z = zj;
    }
    loss[r] = (t >= 0 && t < V) ? tot.m + logf(tot.s) - z : __int_as_float(0x7FC00000);
  }
}

// Row kernels may be launched as programmatic dependents of the kernel before
// them in the stream: their blocks are scheduled while that grid drains and
// wait (griddep_wait, their first statement after allowing their own
// dependents) until it has completed.
template <class... P, class... A>
cudaError_t launch_row_kernel(void (*kernel)(P...), unsigned grid, unsigned block, cudaStream_t st, A&&... args) {
#if LMHO_CE_PDL
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(block);
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<A>(args)...);
#else
  kernel<<<grid, block, 0, st>>>(std::forward<A>(args)...);
  return cudaSuccess;
#endif
}

template <typename T, class Sink>
cudaError_t launch_rows(const T* logits, const int64_t* target, int64_t rows, int64_t V, Sink sink,
                        const float* rows_for_mean, float* mean_out, Ctrl* ctrl, const CeConfig& cfg,
                        cudaStream_t st) {
  launch_mark(0, st);
  cudaError_t le = cudaSuccess;
  switch (cfg.variant) {
    case kCeWarp: {
      // 16 loads per lane in flight: a 16 KB row takes one or two memory round
      // trips, a 32 KB row four (with 4 in flight, 16; Megatron bf16 V = 16384
      // measured 49.3-49.6 vs 50.1-50.2 us, 64 vs 54 registers).  Blocks of 2
      // warps: Megatron V = 16384 47.6-47.9 us against 49.2 with 8 warps, the
      // same at V = 4096 and 8192, one event tick slower with 16.
      // bf16 folds all 16 vectors at once (packed max, then one exponent pass:
      // 31 % fewer instructions than folds of 2 unpacked vectors; 88 registers,
      // 22 warps per SM; Megatron V = 8192 22.9 us against 24.6, V = 16384
      // 42.6 against 45.4).  fp32 folds 4 at a time within 64 registers (16
      // blocks, 32 warps): builds held to 40 or 32 registers spill and were
      // 4-90 % slower.
      // Rows on 16-byte boundaries (every workload size) take an instance
      // without the scalar head and tail: 88 instead of 96 registers for bf16,
      // 11 resident blocks instead of 10.
      const unsigned nb = static_cast<unsigned>((rows + 1) / 2);
      const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (V * sizeof(T)) % 16 == 0;
      if constexpr (sizeof(T) == 2) {
        if (aligned)
          le = launch_row_kernel(ce_warp_rows<T, 16, 16, 1, true, Sink>, nb, 64, st, logits, target, rows, V, sink);
        else
          le = launch_row_kernel(ce_warp_rows<T, 16, 16, 1, false, Sink>, nb, 64, st, logits, target, rows, V, sink);
      } else {
        if (aligned)
          le = launch_row_kernel(ce_warp_rows<T, 16, LMHO_CE_F32_FOLD, 16, true, Sink>, nb, 64, st, logits, target, rows,
                            V, sink);
        else
          le = launch_row_kernel(ce_warp_rows<T, 16, LMHO_CE_F32_FOLD, 16, false, Sink>, nb, 64, st, logits, target, rows,
                            V, sink);
      }
      break;
    }
    case kCeCta:
      if (cfg.threads == 512)
        le = launch_row_kernel(ce_cta_rows<T, 4, 512, Sink>, static_cast<unsigned>(rows), 512, st, logits, target, rows, V,
                          sink);
      else
        le = launch_row_kernel(ce_cta_rows<T, 4, 256, Sink>, static_cast<unsigned>(rows), 256, st, logits, target, rows, V,
                          sink);
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
          ensure_smem_limit(ce_bulk_rows<T, 8, Sink>, static_cast<int>(kCeBulkRingBytes + 128 + 16 * 32), limit_set);
      if (e != cudaSuccess) return e;
      int64_t grid = rows < cfg.num_sms ? rows : cfg.num_sms;
      const int64_t per = (rows + grid - 1) / grid;
      grid = (rows + per - 1) / per;   // no CTA without rows
      ce_bulk_rows<T, 8, Sink><<<static_cast<unsigned>(grid), 32 * 9, smem, st>>>(logits, target, rows, V, sink, ctrl,
                                                                                 stages, nwa, stage_bytes, cfg.timeout_ns);
      break;
    }
    case kCeCluster: {
      const unsigned grid = static_cast<unsigned>(rows * cfg.cluster);
      if (cfg.cluster == 2)
        ce_cluster_rows<T, 4, 256, 2><<<grid, 256, 0, st>>>(logits, target, rows, V, sink);
      else if (cfg.cluster == 4)
        ce_cluster_rows<T, 4, 256, 4><<<grid, 256, 0, st>>>(logits, target, rows, V, sink);
      else
        ce_cluster_rows<T, 4, 256, 8><<<grid, 256, 0, st>>>(logits, target, rows, V, sink);
      break;
    }
    default:
      return cudaErrorInvalidValue;
  }
  if (le != cudaSuccess) return le;
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  if (mean_out) {
    // The mean: one block behind the row kernel, allowed to launch before the
    // row kernel completes (programmatic stream serialization); it waits for
    // that grid's completion in-kernel.  No event may sit between the two
    // kernels, or the overlap is lost: the call's events bracket both.
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
    if (const cudaError_t e = cudaLaunchKernelEx(&lc, ce_mean_rows, rows_for_mean, rows, mean_out); e != cudaSuccess)
      return e;
  }
  launch_mark(1, st);
  return cudaGetLastError();
}

// Bare read of `nseg` segments of `seg_vec` 16-byte vectors with the access of
// the warp-per-row kernel (two-warp blocks, a warp per segment, 16 loads per
// lane in flight, coalesced), folding nothing but an XOR per segment: the
// read-once floor a cross-entropy call over rows of that size can approach.
__global__ void __launch_bounds__(64, 16) probe_read_rows(const uint4* __restrict__ data, int64_t nseg,
                                                          int64_t seg_vec, uint32_t* __restrict__ out) {
  // launched like the CE row kernels (programmatic dependent), so back-to-back
  // probes compare with back-to-back calls
  griddep_launch_dependents();
#if LMHO_CE_PDL
  griddep_wait();
#endif
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 2 + (threadIdx.x >> 5);
  if (r >= nseg) return;
  const uint4* row = data + r * seg_vec;
  uint32_t acc = 0;
  for (int64_t q0 = 0; q0 < seg_vec; q0 += 32 * 16) {
    uint4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int64_t q = q0 + u * 32 + lane;
      v[u] = q < seg_vec ? ldg_stream_v4(row + q) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) out[r] = acc;
}

}  // namespace

cudaError_t launch_ce_f32(const float* logits, const int64_t* target, int64_t T, int64_t V,
                          float* loss, float* row_loss, Ctrl* ctrl, const CeConfig& cfg,
                          cudaStream_t st) {
  return launch_rows<float>(logits, target, T, V, LossSink{row_loss}, row_loss, loss, ctrl, cfg, st);
}

cudaError_t launch_ce_bf16_rows(const uint16_t* logits, const int64_t* target, int64_t rows,
                                int64_t V, float* loss_rows, const CeConfig& cfg, cudaStream_t st) {
  return launch_rows<uint16_t>(logits, target, rows, V, LossSink{loss_rows}, nullptr, nullptr, nullptr, cfg, st);
}

cudaError_t launch_ce_partials_bf16(const uint16_t* logits, const int64_t* target, int64_t rows, int64_t V_local,
                                    int64_t v0, float* partials, const CeConfig& cfg, cudaStream_t st) {
  const PartialSink sink{partials, partials + rows, partials + 2 * rows, v0};
  return launch_rows<uint16_t>(logits, target, rows, V_local, sink, nullptr, nullptr, nullptr, cfg, st);
}

cudaError_t launch_ce_partials_f32(const float* logits, const int64_t* target, int64_t rows, int64_t V_local,
                                   int64_t v0, float* partials, const CeConfig& cfg, cudaStream_t st) {
  const PartialSink sink{partials, partials + rows, partials + 2 * rows, v0};
  return launch_rows<float>(logits, target, rows, V_local, sink, nullptr, nullptr, nullptr, cfg, st);
}

cudaError_t launch_probe_read(const void* data, int64_t nseg, int64_t seg_bytes, uint32_t* out, cudaStream_t st) {
  launch_mark(0, st);
  const unsigned nb = static_cast<unsigned>((nseg + 1) / 2);
  const cudaError_t e = launch_row_kernel(probe_read_rows, nb, 64, st, static_cast<const uint4*>(data), nseg,
                                          seg_bytes / 16, out);
  if (e != cudaSuccess) return e;
  launch_mark(1, st);
  return cudaGetLastError();
}

cudaError_t launch_ce_merge(const float* partials, int64_t shards, const int64_t* target, int64_t rows, int64_t V,
                            float* loss, int num_sms, cudaStream_t st) {
  launch_mark(0, st);
  int64_t blocks = (rows + 255) / 256;
  if (blocks > 8 * static_cast<int64_t>(num_sms)) blocks = 8 * static_cast<int64_t>(num_sms);
  ce_merge_rows<<<static_cast<unsigned>(blocks), 256, 0, st>>>(partials, shards, target, rows, V, loss);
  launch_mark(1, st);
  return cudaGetLastError();
}

}  // namespace lmho
