// Combinations of vocabulary shards' per-token results for the vocab-parallel
// fused losses (page "Vocab-parallel cross-entropy, Megatron layout", summary:
// each tensor-parallel rank holds its own vocab range; here that split applied
// to the rows of the output layer W, page "Fused linear + JSD" for the
// divergence), and the deterministic mean of per-token values.
//
//   * log-sum-exp merge: each head's global log-sum-exp of token i from the
//     shards' own, l_j, in shard order: L = max_j l_j, lse = L + ln sum_j
//     exp(l_j - L) (a NaN propagates);
//   * JSD term merge: token i's divergence is the sum, in shard order, of the
//     shards' sums of its JSD terms (compensated fp32); tokens whose keep
//     flag is 0 get 0; then the batchmean over the kept tokens;
//   * row mean: fixed-order compensated fp32 mean of per-token values (over
//     the kept ones when a mask is given), bitwise reproducible;
//   * the global log-sum-exp of each token from gathered cross-entropy
//     partials, for the backward of the vocab-parallel fused CE.
// The cross-entropy's shard merge is ce_merge_rows (ce_rows.cu).
//
// All of them are tiny next to the passes that produce their inputs: they read
// 8 k or 4 k bytes per token for k shards.
#include <cmath>
#include <cstdint>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace lmho {
namespace {

// lse [2][T] from parts [k][2][T] (shard-major): one thread per (head, token).
__global__ void __launch_bounds__(256) lse_merge_rows(const float* __restrict__ parts, int64_t shards, int64_t T,
                                                       float* __restrict__ lse) {
  const int64_t n = 2 * T;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // q = head * T + token; shard j's value sits at parts[j * 2T + q]
    float L = __ldg(parts + q);
    for (int64_t j = 1; j < shards; ++j) {
      const float l = __ldg(parts + j * n + q);
      if (l > L || l != l) L = l;
    }
    float sum = 0.f;
    for (int64_t j = 0; j < shards; ++j) sum += expf(__ldg(parts + j * n + q) - L);
    lse[q] = L + logf(sum);
  }
}

// rows [T] from terms [k][T]: the shards' sums in shard order, compensated.
// Lets its dependent (the mean) launch at once.
__global__ void __launch_bounds__(256) jsd_merge_rows(const float* __restrict__ terms, int64_t shards, int64_t T,
                                                       const uint8_t* __restrict__ keep, float* __restrict__ rows) {
  griddep_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < T;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    KSum a;
    for (int64_t j = 0; j < shards; ++j) a.add(__ldg(terms + j * T + i));
    rows[i] = (keep && !__ldg(keep + i)) ? 0.f : a.s - a.c;
  }
}

// Mean of rows [T] (over the kept ones when keep is set; 0 when none is
// kept), one block of 256 threads.  As a programmatic dependent of the kernel
// that wrote the rows, griddep_wait() returns once that grid has completed
// and its writes are visible; launched alone it returns at once.
__global__ void __launch_bounds__(256) rows_mean_kernel(const float* __restrict__ rows, int64_t T,
                                                         const uint8_t* __restrict__ keep, float* __restrict__ mean) {
  griddep_wait();
  mean_sum(rows, T, mean, keep);
}

// lse [T] from gathered cross-entropy partials [k][3][T] (m, s, z per shard):
// the (m, s) merged in shard order exactly as ce_merge_rows merges them, then
// m + ln s -- each token's global log-sum-exp, for the sharded backward.
__global__ void __launch_bounds__(256) partials_lse_rows(const float* __restrict__ part, int64_t shards, int64_t T,
                                                          float* __restrict__ lse) {
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < T;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    MS tot = ms_empty();
    for (int64_t j = 0; j < shards; ++j) {
      const float* p = part + 3 * j * T;
      tot = ms_merge(tot, MS{__ldg(p + r), __ldg(p + T + r)});
    }
    lse[r] = tot.m + logf(tot.s);
  }
}

// 1 / (number of tokens with keep != 0), or 1 / T with no mask, 0 when none is
// kept: one block, an exact integer count in a fixed order.
__global__ void __launch_bounds__(256) kept_inv_count_kernel(const uint8_t* __restrict__ keep, int64_t T,
                                                              float* __restrict__ inv_count) {
  __shared__ int64_t s_cnt[256];
  int64_t c = 0;
  if (keep) {
    for (int64_t i = threadIdx.x; i < T; i += 256) c += __ldg(keep + i) != 0;
  } else {
    for (int64_t i = threadIdx.x; i < T; i += 256) ++c;
  }
  s_cnt[threadIdx.x] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t n = 0;
    for (int k = 0; k < 256; ++k) n += s_cnt[k];
    *inv_count = n > 0 ? 1.f / static_cast<float>(n) : 0.f;
  }
}

unsigned grid_for(int64_t n, int num_sms) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8 * static_cast<int64_t>(num_sms)) blocks = 8 * static_cast<int64_t>(num_sms);
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_lse_merge(const float* parts, int64_t shards, int64_t T, float* lse, int num_sms,
                             cudaStream_t st) {
  launch_mark(0, st);
  lse_merge_rows<<<grid_for(2 * T, num_sms), 256, 0, st>>>(parts, shards, T, lse);
  launch_mark(1, st);
  return cudaGetLastError();
}

cudaError_t launch_jsd_merge(const float* terms, int64_t shards, int64_t T, const uint8_t* keep, float* rows,
                             float* loss, int num_sms, cudaStream_t st) {
  launch_mark(0, st);
  jsd_merge_rows<<<grid_for(T, num_sms), 256, 0, st>>>(terms, shards, T, keep, rows);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
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
  if (const cudaError_t e = cudaLaunchKernelEx(&lc, rows_mean_kernel, static_cast<const float*>(rows), T, keep, loss);
      e != cudaSuccess)
    return e;
  launch_mark(1, st);
  return cudaGetLastError();
}

cudaError_t launch_partials_lse(const float* partials, int64_t shards, int64_t T, float* lse, int num_sms,
                                cudaStream_t st) {
  partials_lse_rows<<<grid_for(T, num_sms), 256, 0, st>>>(partials, shards, T, lse);
  return cudaGetLastError();
}

cudaError_t launch_kept_inv_count(const uint8_t* keep, int64_t T, float* inv_count, cudaStream_t st) {
  kept_inv_count_kernel<<<1, 256, 0, st>>>(keep, T, inv_count);
  return cudaGetLastError();
}

cudaError_t launch_rows_mean(const float* rows, int64_t n, const uint8_t* keep, float* mean, cudaStream_t st) {
  launch_mark(0, st);
  rows_mean_kernel<<<1, 256, 0, st>>>(rows, n, keep, mean);
  launch_mark(1, st);
  return cudaGetLastError();
}

}  // namespace lmho
