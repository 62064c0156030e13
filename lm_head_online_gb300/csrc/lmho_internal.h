// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lmho {

// Raises `kern`'s dynamic shared-memory limit to `bytes` on the current device,
// once per device per call site (`done`: the site's static per-device flags).
// Safe to call from several host threads: the flags are atomic, and two first
// calls that race both set the same attribute.
constexpr int kMaxDevices = 64;
template <class K>
cudaError_t ensure_smem_limit(K kern, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
  return e;
}

struct Ctrl;

// ---------------------------------------------------------------- CE rows
enum CeVariant { kCeWarp = 0, kCeCta = 1, kCeCluster = 2, kCeBulk = 3 };
struct CeConfig {
  int variant;          // CeVariant
  int threads;          // CTA size of the CTA-per-row kernel (256 or 512)
  int cluster;          // CTAs per row of the cluster kernel (2, 4 or 8)
  int num_sms = 0;      // bulk kernel: one persistent CTA per SM
  uint64_t timeout_ns = 2000000000ull;  // bulk kernel: bound of every mbarrier wait
  uint32_t bulk_ring_bytes = 0;         // bulk kernel: ring size (0 = kCeBulkRingBytes)
};

// Row decomposition of a cross-entropy call over `rows` rows of V elements of
// `elt` bytes starting at `base` (the automatic rule, or the process-wide
// override of lmho_set_ce_variant).
CeConfig choose_ce(const void* base, int64_t rows, int64_t V, size_t elt, int num_sms);

// Largest row (bytes) the bulk-copy ring kernel takes: two stages must fit.
constexpr uint32_t kCeBulkRingBytes = 200 * 1024;
constexpr uint32_t kCeBulkMaxRow = kCeBulkRingBytes / 2;

cudaError_t launch_ce_f32(const float* logits, const int64_t* target, int64_t T, int64_t V,
                          float* loss, float* row_loss, Ctrl* ctrl, const CeConfig& cfg,
                          cudaStream_t st);
cudaError_t launch_ce_bf16_rows(const uint16_t* logits, const int64_t* target, int64_t rows,
                                int64_t V, float* loss_rows, const CeConfig& cfg, cudaStream_t st);

// Vocab-parallel cross-entropy: one shard's partials (max, sum of exp,
// target logit or -inf) of bf16 rows [rows, V_local] holding the global
// columns [v0, v0 + V_local), written as [3][rows] floats; and the merge of
// `shards` such blocks ([shards][3][rows]) into per-row losses.
cudaError_t launch_ce_partials_bf16(const uint16_t* logits, const int64_t* target, int64_t rows, int64_t V_local,
                                    int64_t v0, float* partials, const CeConfig& cfg, cudaStream_t st);
// The same for fp32 logits [rows, V_local] (the flat layout).
cudaError_t launch_ce_partials_f32(const float* logits, const int64_t* target, int64_t rows, int64_t V_local,
                                   int64_t v0, float* partials, const CeConfig& cfg, cudaStream_t st);
cudaError_t launch_ce_merge(const float* partials, int64_t shards, const int64_t* target, int64_t rows, int64_t V,
                            float* loss, int num_sms, cudaStream_t st);

// Bandwidth probe: `nseg` segments of seg_bytes (a multiple of 16) read with
// the warp-per-row kernel's loads; one XOR word per segment to out.
cudaError_t launch_probe_read(const void* data, int64_t nseg, int64_t seg_bytes, uint32_t* out, cudaStream_t st);

// Forward + backward (loss and gradient w.r.t. the logits), one HBM pass.
// gscale: gradient weight per row (flat: grad_scale / T; per-token rows also
// multiplied by dloss[r] when dloss is non-null).
cudaError_t launch_ce_fwd_bwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V, float gscale,
                                  float* loss, float* row_loss, float* dlogits, Ctrl* ctrl, uint64_t timeout_ns,
                                  cudaStream_t st);
cudaError_t launch_ce_fwd_bwd_bf16_rows(const uint16_t* logits, const int64_t* target, int64_t rows, int64_t V,
                                        const float* dloss, float gscale, float* loss_rows, uint16_t* dlogits,
                                        uint64_t timeout_ns, cudaStream_t st);

// ---------------------------------------------------------------- fused linear
// Tile geometry of the tensor-core kernels.
constexpr int kBM = 128;        // token rows per tile (TMEM lanes)
constexpr int kBK = 64;         // hidden elements per pipeline stage (one 128-byte swizzle row)
constexpr int kBN_CE = 256;     // vocab columns per tile, single-head passes
#ifndef LMHO_JSD_BN
#define LMHO_JSD_BN 256
#endif
constexpr int kBN_JSD = LMHO_JSD_BN;  // vocab columns per head per tile, two-head pass
constexpr int kJsdColSplit = 2;       // two-head pass: epilogue warps per TMEM lane quadrant
// CTA pairs (tcgen05 cta_group::2): a unit is a tile of 2 x kBM rows by kBN_CE
// columns, each CTA of the pair loading its kBM rows of A and half of B
// (kBN_CE / 2 rows of the N extent) and holding its kBM rows of the
// accumulator.  The gradient products (dx = dZ W, dW = dZ^T x) run on pairs:
// their MN-major operands are feed-bound on a lone CTA, and a pair's SM loads
// 2/3 of the operand bytes per k-block (dW 11 %, dx 9 % faster in short
// calls, both 7 % in 40 ms power-capped ones).  The CE, log-sum-exp and dZ
// passes run on lone CTAs
// (M = 128): paired they are ~5 % faster in short calls but 3-5 % slower
// under the power cap, where they spend most of their time.  LMHO_PAIR_FWD /
// LMHO_PAIR_GRAD (0 or 1) choose at build time; kBoxBFwd / kBoxBGrad are the
// B rows one CTA loads (the host's tensor-map boxes).
#ifndef LMHO_PAIR_FWD
#define LMHO_PAIR_FWD 0
#endif
#ifndef LMHO_PAIR_GRAD
#define LMHO_PAIR_GRAD 1
#endif
constexpr bool kPairFwd = LMHO_PAIR_FWD != 0;    // CE, log-sum-exp, dZ passes
constexpr bool kPairGrad = LMHO_PAIR_GRAD != 0;  // dx, dW
constexpr int kBoxBFwd = kPairFwd ? kBN_CE / 2 : kBN_CE;
constexpr int kBoxBGrad = kPairGrad ? kBN_CE / 2 : kBN_CE;
// MN-major operands move in 128-byte rows of 64 bf16 ("chunks").  When the MN
// extent is a whole number of chunks the tensor map is 3-D (64 elements, K rows,
// chunks) and one TMA copy fills a whole tile's operand; otherwise it is 2-D and
// a tile takes one copy per chunk, the map's edge zero-filling the ragged one.
constexpr int kMnChunk = 64;
inline bool mn_chunked(int64_t mn) { return mn % kMnChunk == 0; }

struct FusedGeometry {
  int64_t T, H, V;
  int64_t num_m, num_n;   // tiles along tokens and vocab
  int group_m;            // m-tiles per raster group (L2 reuse of W)
  int group_store;        // raster group of the gradient products (dx, dW)
};
// Default raster groups (token tiles of 128): single-head passes keep 32 tiles'
// x and the W tiles a wave shares in L2; a two-head pass holds both heads' tiles,
// so half as many; the gradient products use 16.  Measured in the power-capped
// bench step: 16 -> 32 took the flce and log-sum-exp passes 1-2 % faster and
// the two-head pass 3 % slower; 64 and 128 thrash L2 (8-15 % slower).
constexpr int kGroupSingle = 32;
constexpr int kGroupTwoHead = 16;
constexpr int kGroupStore = 16;

// Workspace carve-up of the fused paths (all offsets 256-byte aligned).
struct FusedWs {
  float* row_out;     // [T] per-token loss / JSD (first bytes of ws, documented)
  float* part0;       // [heads][num_n][T]  running max, or JSD partial sums
  float* part1;       // [heads][num_n][T]  running sum of exp
  float* part2;       // [num_n][T]         target logit (CE) / unused
  float* lse;         // [2][T]             log-sum-exp of student, teacher (JSD)
  Ctrl* ctrl;         // last 256 bytes
};

size_t flce_ws_bytes(int64_t T, int64_t H, int64_t V);
size_t fljsd_ws_bytes(int64_t T, int64_t H, int64_t V);
FusedWs flce_ws_carve(void* ws, size_t ws_bytes, int64_t T, int64_t V);
FusedWs fljsd_ws_carve(void* ws, size_t ws_bytes, int64_t T, int64_t V);

struct FusedLaunch {
  int num_sms;
  uint64_t timeout_ns;
  cudaStream_t stream;
};

// x [T,H], W [V,H] -> loss[1]; tensor maps built by the caller.
cudaError_t launch_flce(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target,
                        const FusedGeometry& g, float* loss, const FusedWs& ws,
                        const FusedLaunch& L);
// Student/teacher head maps come twice: 256-row boxes for the log-sum-exp
// pass and kBN_JSD-row boxes for the two-head divergence pass.
cudaError_t launch_fljsd(const CUtensorMap& tm_xs, const CUtensorMap& tm_ws256,
                         const CUtensorMap& tm_xt, const CUtensorMap& tm_wt256,
                         const CUtensorMap& tm_wsj, const CUtensorMap& tm_wtj,
                         const FusedGeometry& g_lse, const FusedGeometry& g_jsd, float beta,
                         float inv_tau, const uint8_t* keep, float* loss, const FusedWs& ws,
                         const FusedLaunch& L);

// Vocab-parallel fused losses, one shard of W's rows (the global vocab
// columns [v0, v0 + g.V)):
//  * fused linear + CE: each token's (max, sum of exp, target logit or -inf)
//    over the shard -> partials [3][T] (m, s, z);
cudaError_t launch_flce_partials(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target, int64_t v0,
                                 const FusedGeometry& g, float* partials, const FusedWs& ws, const FusedLaunch& L);
//  * fused linear + JSD, first pass: each head's log-sum-exp of logits / tau
//    over the shard -> lse_local [2][T];
cudaError_t launch_fljsd_lse_shard(const CUtensorMap& tm_xs, const CUtensorMap& tm_ws256, const CUtensorMap& tm_xt,
                                   const CUtensorMap& tm_wt256, const FusedGeometry& g_lse, float inv_tau,
                                   float* lse_local, const FusedWs& ws, const FusedLaunch& L);
//  * fused linear + JSD, second pass: with the global log-sum-exps lse [2][T],
//    each token's sum of the JSD terms over the shard's columns -> terms [T].
//    With kl_local set, also each token's share of KL(P || M) over the shard
//    -> kl_local [T] (the backward's variant; the same divergence bits).
cudaError_t launch_fljsd_terms_shard(const CUtensorMap& tm_xs, const CUtensorMap& tm_wsj, const CUtensorMap& tm_xt,
                                     const CUtensorMap& tm_wtj, const FusedGeometry& g_jsd, const float* lse,
                                     float beta, float inv_tau, float* terms, float* kl_local, const FusedWs& ws,
                                     const FusedLaunch& L);
// Their combinations (vp_merge.cu): global log-sum-exps [2][T] from k shards'
// [k][2][T]; per-token JSD rows [T] and their batchmean from k shards' term
// sums [k][T] (keep may be null); and the deterministic mean of n values
// (16-byte aligned) over the kept ones.
cudaError_t launch_lse_merge(const float* parts, int64_t shards, int64_t T, float* lse, int num_sms,
                             cudaStream_t st);
cudaError_t launch_jsd_merge(const float* terms, int64_t shards, int64_t T, const uint8_t* keep, float* rows,
                             float* loss, int num_sms, cudaStream_t st);
cudaError_t launch_rows_mean(const float* rows, int64_t n, const uint8_t* keep, float* mean, cudaStream_t st);
// 1 / (kept tokens) (keep may be null: 1 / T; 0 when none is kept) -> inv_count [1].
cudaError_t launch_kept_inv_count(const uint8_t* keep, int64_t T, float* inv_count, cudaStream_t st);
// Each token's global log-sum-exp [T] from gathered CE partials [k][3][T].
cudaError_t launch_partials_lse(const float* partials, int64_t shards, int64_t T, float* lse, int num_sms,
                                cudaStream_t st);

// Records the caller's measurement event `i` on `st` if the hook is set
// (lmho_set_launch_events); no-op otherwise.
void launch_mark(int i, cudaStream_t st);

// Fused linear + CE forward and backward.  Workspace beyond the forward's:
// each row's log-sum-exp, dZ (bf16 [T, ld_dz], ld_dz a multiple of 256) and,
// when a gradient product has too few output tiles to fill the machine, fp32
// K slices of it (kMaxKSplit x its size) for a split-K product.
struct FlceBwdWs {
  float* lse;
  uint16_t* dz;
  float* split;   // null when neither product can split
  int64_t ld_dz;
};
// Split-K of the gradient products dx = dZ W and dW = dZ^T x: only below
// kSplitTiles output tiles of 128 x 256 (a pair's 256-row tile counts as two),
// into at most kMaxKSplit slices of at least kMinSplitKBlocks k-blocks each.
constexpr int64_t kSplitTiles = 4 * 152;
constexpr int kMaxKSplit = 8;
constexpr int kMinSplitKBlocks = 16;
// Bytes of fp32 slices a product with an [M, N] output may need (0 = never splits).
size_t k_split_reserve_bytes(int64_t M, int64_t N);
// K slices for `tiles` output tiles and `k_blocks` k-blocks on `num_sms` SMs.
int choose_k_split(int64_t tiles, int k_blocks, int num_sms);

// Tensor maps of the backward.  K-major maps have boxes of 64 (K) x rows;
// MN-major maps (_mn) cover a [K, MN] matrix with boxes of 64 (MN) x 64 (K).
struct FlceBwdMaps {
  CUtensorMap x, w;      // forward and dZ passes: A = x [T, H], B = W [V, H]
  CUtensorMap dz, w_mn;  // dx = dZ W:   A = dZ [T, V] (K = V), B = W [V, H] MN-major
  CUtensorMap dz_mn, x_mn;  // dW = dZ^T x: A = dZ [T, V] MN-major (K = T), B = x [T, H] MN-major
};
size_t flce_bwd_ws_bytes(int64_t T, int64_t H, int64_t V);
FlceBwdWs flce_bwd_ws_carve(void* ws, int64_t T, int64_t H, int64_t V);
// Fused linear + CE backward of one vocabulary shard (W = the global rows
// [v0, v0 + g.V)): each token's global log-sum-exp from the gathered CE
// partials [shards][3][T] (into bw.lse), the shard's dZ columns (targets global; v_total = the global vocabulary
// size), this shard's share of dx (the ranks' shares sum to dx) and its own
// rows of dW.
// Row weights: null = the mean's grad_scale / T on every row, else
// grad_scale * row_w[i] (e.g. CPO's d loss / d l_i).
cudaError_t launch_flce_shard_bwd(const FlceBwdMaps& m, const int64_t* target, const float* partials,
                                  int64_t shards, int64_t v0, int64_t v_total, const FusedGeometry& g,
                                  float grad_scale, const float* row_w, float* dx, float* dW, const FusedWs& ws,
                                  const FlceBwdWs& bw, const FusedLaunch& L);
// CPO on the fused linear + CE: pairs of sequences (chosen b, rejected b + B/2)
// of S tokens.  Workspace pieces beyond the fused CE's.
struct CpoArgs {
  int64_t B, S;
  float beta, alpha;
  float* lp;      // [B]   sequence log-likelihoods
  float* sig;     // [B/2] sigmoid(-beta d_k)
  float* mean;    // [1]   the token mean the CE finaliser writes (not the CPO loss)
  float* logps;   // [B]   caller copy of lp, or null
  float* row_w;   // [T]   backward: d loss / d l_i, or null
};
// The CPO combination of given per-token CE losses rows [B * S]: loss, the
// sequence log-likelihoods (logps, may be null) and, with row_w set, each
// token's weight d loss / d l_i; lp [B], sig [B / 2] scratch, ctrl->ticket 0.
cudaError_t launch_cpo_combine(const float* rows, int64_t B, int64_t S, float beta, float alpha, float* loss,
                               float* logps, float* row_w, float* lp, float* sig, Ctrl* ctrl, cudaStream_t st);
cudaError_t launch_flce_cpo(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target,
                            const FusedGeometry& g, float* loss, const FusedWs& ws, const CpoArgs& c,
                            const FusedLaunch& L);
// With `cpo` set the loss is the CPO objective and dZ carries its per-row weights.
cudaError_t launch_flce_fwd_bwd(const FlceBwdMaps& m, const int64_t* target, const FusedGeometry& g, float grad_scale,
                                float* loss, float* dx, float* dW, const FusedWs& ws, const FlceBwdWs& bw,
                                const FusedLaunch& L, const CpoArgs* cpo = nullptr);

// Fused linear + JSD forward and student backward.
struct FljsdBwdMaps {
  CUtensorMap xs, xt, ws256, wt256, wsj, wtj;  // the forward passes, and the dZ pass
  CUtensorMap dz, ws_mn;                        // dxs = dZs Ws
  CUtensorMap dz_mn, xs_mn;                     // dWs = dZs^T xs
};
size_t fljsd_bwd_ws_bytes(int64_t T, int64_t H, int64_t V);
// Student backward of one vocabulary shard of the fused linear + JSD: with the
// global log-sum-exps lse [2][T] and KL(P || M) kl [T] (the shards' shares
// summed), the shard's dZs columns, its share of dxs and its rows of dWs.
cudaError_t launch_fljsd_shard_bwd(const FljsdBwdMaps& m, const FusedGeometry& g_jsd, float beta, float inv_tau,
                                   const uint8_t* keep, float grad_scale, const float* lse, const float* kl,
                                   float* dxs, float* dWs, const FusedWs& ws, const FlceBwdWs& bw, float* inv_count,
                                   const FusedLaunch& L);
cudaError_t launch_fljsd_fwd_bwd(const FljsdBwdMaps& m, const FusedGeometry& g_lse, const FusedGeometry& g_jsd,
                                 float beta, float inv_tau, const uint8_t* keep, float grad_scale, float* loss,
                                 float* dxs, float* dWs, const FusedWs& ws, const FlceBwdWs& bw, float* kl,
                                 float* inv_count, const FusedLaunch& L);

cudaError_t launch_wait_selftest(Ctrl* ctrl, uint64_t timeout_ns, cudaStream_t st);

}  // namespace lmho
