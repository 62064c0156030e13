// Fused linear + cross-entropy, + CPO and + generalized JSD on the
// 5th-generation tensor cores, forward and backward, logits never written to
// memory.
//
// Operations: page "Fused linear + CPO loss" (summary: activations projected
// through a vocab x hidden LM head, "computed chunked without materializing
// logits"; Semantics: x, weight, target, loss) and page "Fused linear + JSD"
// (summary: student and teacher heads, generalized JSD with beta 0.5,
// batchmean).
//
// One persistent kernel per pass, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: bf16 tiles of A [128 x 64] and B [rows x 64]
//               (128-byte swizzle; K-major, or MN-major 64 x 64 boxes for the
//               gradient products, one 3-D copy per tile where the MN extent is
//               whole 64-element chunks) into a ring of shared-memory stages
//               (mbarrier complete_tx);
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (K=16, bf16 x bf16 -> fp32) and frees stages with
//               tcgen05.commit;
//   warps 2..   epilogue (4 warps, 8 for the two-head passes): each thread owns
//               one token row (one TMEM lane) and reads its accumulator row with
//               tcgen05.ld.
// The gradient products (STORE) run on CTA pairs, clusters of 2 with tcgen05
// cta_group::2: a unit is 256 rows x 256 columns, each CTA loads its 128 rows of
// A and 128 of the 256 rows of B (a pair reads 2/3 of the operand bytes two lone
// CTAs would), the even CTA issues M=256 N=256 MMAs for both, and each CTA's
// TMEM holds its 128 rows of D.  The other single-head passes (CE, LSE, DZ) run
// on lone CTAs, M=128 N=256 (which passes pair is a build-time choice).  Both
// double-buffer two 256-column accumulators, so the epilogue of one unit
// overlaps the MMAs of the next.  Two-head passes (JSD, JSDK, DZJ; BN = 256 per
// head) run on lone CTAs: one unit fills TMEM, its heads complete and are
// released separately, so the next unit's student MMAs overlap this unit's
// epilogue.
// Work unit = (token tile, vocab tile), rastered in groups of `group_m` token
// tiles so a wave of CTAs shares the same W tiles in L2 and each W tile is
// read from HBM about once per group.
//
// Epilogues (per row r of the tile, vocab columns n0 .. n0+BN-1):
//   CE     running (max, sum exp) of the tile and the target logit if t_r
//          falls in the tile  -> partials [num_n][T] x 3
//   LSE    (max, sum exp) only, for the student and teacher heads (first JSD
//          pass)  -> partials [2][num_n][T] x 2
//   JSD    both heads' tiles; the generalized-JSD term of every pair, evaluated
//          around the larger log-probability so no large terms cancel
//          -> partial sums [num_n][T] (JSDK: also KL(P || M) for the backward)
//   DZ     the CE gradient of the tile, bf16 dZ rows (DZJ: the JSD student's)
//   STORE  fp32 tile of a gradient product (dx = dZ W, dW = dZ^T x)
// Finalisers merge the vocab-tile partials of each row in a fixed order and
// reduce the rows deterministically (see rowstats.cuh).
#include <cmath>
#include <cstdint>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

#ifndef LMHO_JSD_PACKED
#define LMHO_JSD_PACKED 1
#endif
#ifndef LMHO_FOLD_PACKED
#define LMHO_FOLD_PACKED 1
#endif

namespace lmho {
namespace {

// CE / LSE / JSD: loss epilogues.  DZ: gradient of the CE with respect to the
// logits, written as bf16 dZ [T, ld_dz] (the operand of both backward GEMMs).
// STORE / STORET: plain fp32 tile store, rows = T and columns = V in Params, of
// the backward GEMMs  dx = dZ W  (STORE: A = dZ K-major, B = W read MN-major)
// and  dW = dZ^T x  (STORET: A = dZ and B = x, both read MN-major), optionally
// split along K into fp32 slices.  JSDK: the divergence pass that also sums
// KL(P || M) per row (backward only).  DZJ: both heads recomputed, the
// student's gradient dZs written like DZ.
enum Mode {
  kModeCE = 0, kModeLSE = 1, kModeJSD = 2, kModeDZ = 3, kModeStore = 4, kModeJSDK = 5, kModeDZJ = 6, kModeStoreT = 7
};

template <int MODE>
constexpr bool two_head() { return MODE == kModeJSD || MODE == kModeJSDK || MODE == kModeDZJ; }
template <int MODE>
constexpr bool store_mode() { return MODE == kModeStore || MODE == kModeStoreT; }
// Operands stored MN-major in global memory ([K, M] / [K, N], M or N contiguous).
template <int MODE>
constexpr bool a_mn() { return MODE == kModeStoreT; }
template <int MODE>
constexpr bool b_mn() { return store_mode<MODE>(); }
constexpr int kMnBox = kMnChunk;                // MN extent of one 128-byte swizzle row of bf16
constexpr int kMnBoxBytes = kMnBox * kBK * 2;   // one TMA box of an MN-major operand: 64 (MN) x 64 (K)

constexpr int kTmemCols = 512;   // all of TMEM: accumulators of 256 or 512 fp32 columns
constexpr int kSmemBudget = 192 * 1024;

template <int MODE>
struct ModeCfg {
  static constexpr int BN = two_head<MODE>() ? kBN_JSD : kBN_CE;
  // CTA pair (single-head passes): a unit is kRowsM = 2 kBM rows; this CTA loads
  // kBM rows of A and kBRows = BN / 2 of B and holds kBM rows of the accumulator.
  static constexpr bool kPair = two_head<MODE>() ? false : store_mode<MODE>() ? kPairGrad : kPairFwd;
  static constexpr int kRowsM = kPair ? 2 * kBM : kBM;
  static constexpr int kBRows = kPair ? BN / 2 : BN;
  static constexpr int kHeadsPerUnit = two_head<MODE>() ? 2 : 1;
  static constexpr int kAccCols = BN * kHeadsPerUnit;      // TMEM columns of one accumulator
  static constexpr int kNumAcc = kTmemCols / kAccCols;     // 2 = double-buffered, 1 = single
  // Full and release barriers: one per accumulator, or one per head of the
  // single two-head accumulator (its heads complete and are freed separately).
  static constexpr int kNumFree = two_head<MODE>() ? 2 : kNumAcc;
  // Epilogue warps: 4 cover the 128 TMEM lanes; 8 = two per lane quadrant,
  // each taking half of the columns (the two-head epilogue is the heavier one).
  static constexpr int kEpiWarps = two_head<MODE>() ? 4 * kJsdColSplit : 4;
  static constexpr int kColSplit = kEpiWarps / 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;    // producer warp, MMA warp, epilogue
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  // STORE epilogues stage each warp's 32 x 32 fp32 block (rows padded to 36
  // floats) to write it back as whole 128-byte rows.
  // The DZ epilogue stages each warp's bf16 rows (32 x 64 bytes, 16-byte chunks
  // XOR-swizzled) the same way.
  static constexpr int kOutPitch = 36;
  static constexpr int kOutStageBytes = store_mode<MODE>() ? kEpiWarps * 32 * kOutPitch * 4
                                        : MODE == kModeDZ ? kEpiWarps * 32 * 64
                                                          : 0;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 512 /*barriers*/ + kOutStageBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kNumAcc >= 1 && kNumAcc * kAccCols == kTmemCols, "accumulators tile TMEM");
  static_assert(BN % (32 * kColSplit) == 0, "epilogue column split");
  // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
  // (bits 7-9 = 1, bits 10-12 = 1), operand majorness in bits 15 (A) and 16 (B),
  // 0 = K-major, 1 = MN-major; N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (a_mn<MODE>() ? 1u << 15 : 0u) |
                                     (b_mn<MODE>() ? 1u << 16 : 0u) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(kRowsM >> 4) << 24);
  static_assert(kBM % kMnBox == 0 && kBRows % kMnBox == 0, "MN-major tiles are whole 64-wide boxes");
  static_assert(two_head<MODE>() || kBRows == (store_mode<MODE>() ? kBoxBGrad : kBoxBFwd),
                "B rows per CTA match the host's tensor-map boxes");
};

struct Params {
  int64_t T, V;
  int32_t num_m, num_n, group_m, k_blocks;
  int64_t units;
  const int64_t* target;  // CE
  int64_t v0;             // CE, DZ: first global vocab column of W (a vocabulary shard; 0 = the whole vocabulary)
  int64_t v_total;        // DZ: global vocabulary size, targets outside [0, v_total) give NaN rows (0 = V)
  float* part0;
  float* part1;
  float* part2;
  const float* lse;  // JSD: [2][T]
  float beta;
  float inv_tau;     // LSE / JSD: logits are multiplied by 1 / temperature
  float gscale;      // DZ: gradient weight of every row (grad_scale / T)
  const float* row_w;  // DZ: per-row factor multiplying gscale (null = 1)
  uint16_t* dz;      // DZ: bf16 [T, ld_dz]
  int64_t ld_dz;
  float* out;        // STORE: fp32 [T, ld_out], or [k_split][T, ld_out] slices
  int64_t ld_out;
  int64_t split_stride;    // STORE: elements between K slices
  int32_t k_split;         // STORE: K slices (units = tiles x k_split)
  int32_t kb_per;          // STORE: k-blocks per slice (the last may be shorter, never empty)
  uint32_t mn3d;           // STORE: bit 0 / bit 1 = the MN-major A / B map is 3-D (one copy per tile)
  const float* kl;         // DZJ: KL(P || M) of every row
  const uint8_t* keep;     // DZJ: token mask (null = all kept)
  const float* inv_count;  // DZJ: 1 / number of kept tokens (device scalar)
  uint64_t timeout_ns;
  uint32_t* status;
};

// Shared-memory descriptor of a K-major bf16 tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart (SBO), start
// address >> 4 in bits 0-13, LBO field 1 (unused for this layout), bits 46-48
// = 0b001, swizzle mode 2 (128-byte) in bits 61-63.  Tiles are 1024-byte
// aligned, so the base-offset field is 0.  Moving 16 bf16 (32 bytes) along K
// inside the swizzle row adds 2 to the start-address field.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// MN-major counterpart of smem_desc_sw128: TMA boxes of 64 (MN) x 64 (K)
// bf16, each K index one 128-byte swizzled row of 64 MN-contiguous elements,
// 8-row swizzle atoms of 1024 bytes.  Canonical MN-major 128-byte-swizzle
// layout: the stride between 8-row groups along K (SBO) is 1024 bytes, the
// stride between 64-element groups along MN (LBO) is one box, 8192 bytes.
// Moving 16 along K advances the start address by 16 rows = 2048 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(kMnBoxBytes >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

struct UnitCoord {
  int head;  // LSE: which head; STORE: which K slice; others 0
  int mt, nt;
};

__device__ __forceinline__ UnitCoord decode_unit(const Params& p, int64_t u, int mode) {
  UnitCoord c{0, 0, 0};
  const int64_t per_head = static_cast<int64_t>(p.num_m) * p.num_n;
  if (mode == kModeLSE || mode == kModeStore || mode == kModeStoreT) {
    c.head = static_cast<int>(u / per_head);
    u -= static_cast<int64_t>(c.head) * per_head;
  }
  const int64_t per_group = static_cast<int64_t>(p.group_m) * p.num_n;
  const int64_t g = u / per_group;
  const int64_t r = u - g * per_group;
  const int64_t m_first = g * p.group_m;
  const int64_t rem = p.num_m - m_first;
  const int64_t gm = rem < p.group_m ? rem : p.group_m;
  c.mt = static_cast<int>(m_first + r % gm);
  c.nt = static_cast<int>(r / gm);
  return c;
}

// Generalized-JSD term of one (token, vocab) pair,
//   beta P (lp - lm) + (1-beta) Q (lq - lm),  lm = ln(beta P + (1-beta) Q),
// from base-2 log-probabilities lp2 = lp log2 e, lq2 = lq log2 e, evaluated
// around the larger side so no large terms cancel: with hi = max(lp2, lq2),
// d = |lp2 - lq2|, (w_hi, w_lo) the beta weights of the larger and smaller
// side, e = 2^-d, u = w_lo e and s = w_hi + u (the argument of the log),
//   hi - lm = -ln2 lg2(s),  lo - lm = -ln2 (lg2(s) + d),
//   term = -ln2 2^hi (s lg2(s) + u d).
// Returns 2^hi (s lg2(s) + u d), the term divided by -ln2 (callers scale the
// sum once): three MUFU operations and no ln2 / log2e multiplies per pair.
// Every step is an explicitly rounded operation (no multiply-add contraction
// left to the compiler), so this and the packed form below give the same bits.
__device__ __forceinline__ float jsd_term2(float lp2, float lq2, float beta, float omb) {
  const float diff = __fsub_rn(lp2, lq2);
  const float hi = fmaxf(lp2, lq2);
  const float d = fabsf(diff);
  const bool p_is_hi = diff >= 0.f;
  const float w_hi = p_is_hi ? beta : omb;
  const float w_lo = p_is_hi ? omb : beta;
  const float u = __fmul_rn(w_lo, ex2_approx(-d));
  const float sv = __fadd_rn(u, w_hi);
  return __fmul_rn(ex2_approx(hi), fmaf(sv, lg2_approx(sv), __fmul_rn(u, d)));
}

// jsd_term2 for two pairs at once (columns j and j + 1 of a row): the FMA,
// subtract, multiply and add steps on packed fp32 pairs (one instruction for
// both), the max / selects and the three MUFU operations per pair unpacked.
// Same arithmetic as jsd_term2; adds the two terms to acc in column order, so
// the row sum is bitwise the one the one-column loops give.
__device__ __forceinline__ void jsd_term2_x2(float& acc, uint64_t zs2, uint64_t zq2, uint64_t it2x2,
                                             uint64_t nls2, uint64_t nlt2, float beta, float omb) {
  float lp0, lp1, lq0, lq1;
  f32x2_split(fma_f32x2(zs2, it2x2, nls2), lp0, lp1);
  f32x2_split(fma_f32x2(zq2, it2x2, nlt2), lq0, lq1);
  float df0, df1;
  f32x2_split(sub_f32x2(f32x2(lp0, lp1), f32x2(lq0, lq1)), df0, df1);
  const float d0 = fabsf(df0), d1 = fabsf(df1);
  const float hi0 = fmaxf(lp0, lq0), hi1 = fmaxf(lp1, lq1);
  const float wh0 = df0 >= 0.f ? beta : omb, wh1 = df1 >= 0.f ? beta : omb;
  const float wl0 = df0 >= 0.f ? omb : beta, wl1 = df1 >= 0.f ? omb : beta;
  float u0, u1;
  f32x2_split(mul_f32x2(f32x2(wl0, wl1), f32x2(ex2_approx(-d0), ex2_approx(-d1))), u0, u1);
  const uint64_t u = f32x2(u0, u1);
  const uint64_t sv = add_f32x2(u, f32x2(wh0, wh1));
  float s0, s1;
  f32x2_split(sv, s0, s1);
  const uint64_t inner = fma_f32x2(sv, f32x2(lg2_approx(s0), lg2_approx(s1)), mul_f32x2(u, f32x2(d0, d1)));
  float t0, t1;
  f32x2_split(mul_f32x2(f32x2(ex2_approx(hi0), ex2_approx(hi1)), inner), t0, t1);
  acc += t0;
  acc += t1;
}

// jsd_term2 and, from the same three MUFU results, the student's pieces the
// KL(P || M) sum needs, in base 2: with lm2 = log2(beta 2^lp2 + (1-beta) 2^lq2)
// = hi + lg2(s),
//   P = 2^lp2 = 2^hi (2^-d when q is the larger side),
//   lp2 - lm2 = -lg2(s) (- d when q is the larger side).
// `term` takes exactly jsd_term2's steps, so the divergence keeps its bits.
__device__ __forceinline__ void jsd_term2_student(float lp2, float lq2, float beta, float omb, float& term, float& P,
                                                  float& lp_lm2) {
  const float diff = __fsub_rn(lp2, lq2);
  const float hi = fmaxf(lp2, lq2);
  const float d = fabsf(diff);
  const bool p_is_hi = diff >= 0.f;
  const float w_hi = p_is_hi ? beta : omb;
  const float w_lo = p_is_hi ? omb : beta;
  const float e = ex2_approx(-d);
  const float u = __fmul_rn(w_lo, e);
  const float sv = __fadd_rn(u, w_hi);
  const float l = lg2_approx(sv);
  const float ph = ex2_approx(hi);
  term = __fmul_rn(ph, fmaf(sv, l, __fmul_rn(u, d)));
  P = p_is_hi ? ph : __fmul_rn(ph, e);
  lp_lm2 = p_is_hi ? -l : -__fadd_rn(l, d);
}

// The pieces of one generalized-JSD pair the backward needs: P = e^{lp} and
// lp - lm (the larger-side evaluation of jsd_term2, in natural log).
__device__ __forceinline__ void jsd_student(float lp, float lq, float beta, float omb, float* P, float* lp_lm) {
  const float hi = fmaxf(lp, lq);
  const float d = fabsf(lp - lq);
  const bool p_is_hi = lp >= lq;
  const float w_hi = p_is_hi ? beta : omb;
  const float w_lo = p_is_hi ? omb : beta;
  const float e = ex2_approx(-d * kLog2e);
  const float a_hi = -kLn2 * lg2_approx(fmaf(w_lo, e, w_hi));
  const float p_hi = ex2_approx(hi * kLog2e);
  *P = p_is_hi ? p_hi : p_hi * e;
  *lp_lm = p_is_hi ? a_hi : a_hi - d;
}

// Two-head epilogue walk over NCH 16-column chunks of this warp's slice of the
// single two-head accumulator: calls f(chunk, student[16], teacher[16]) with
// the fp32 accumulator bits of the warp's 32 rows.  The student head (complete
// when the caller's wait on its full barrier returned) is read into registers
// and its TMEM columns released on free0 while the MMA warp still computes the
// teacher head; once full1 (the teacher head) completes its chunks are read one
// by one, and free1 releases them.  Returns false if the wait on full1 gave up.
template <int NCH, class F>
__device__ __forceinline__ bool two_head_walk(uint32_t tbase, uint32_t head_off, uint64_t* full1, uint32_t parity,
                                              uint64_t* free0, uint64_t* free1, uint64_t timeout_ns,
                                              uint32_t* status, F&& f) {
  uint32_t st[NCH][16], te[16];
#pragma unroll
  for (int c = 0; c < NCH; ++c) tmem_ld16(tbase + c * 16, st[c]);
  tmem_wait_ld(st[0]);
#pragma unroll
  for (int c = 1; c < NCH; ++c) reg_after_wait(st[c]);
  tc_fence_before();
  mbar_arrive(free0);
  if (!__all_sync(0xFFFFFFFFu, mbar_wait(full1, parity, timeout_ns, status))) return false;
  tc_fence_after();
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    tmem_ld16(tbase + head_off + c * 16, te);
    tmem_wait_ld(te);
    f(c, st[c], te);
  }
  tc_fence_before();
  mbar_arrive(free1);
  return true;
}

template <int MODE>
__global__ void __launch_bounds__(ModeCfg<MODE>::kThreads, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_b0,
                      const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_b1,
                      const Params p) {
  using C = ModeCfg<MODE>;
  constexpr int BN = C::BN;
  constexpr int S = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* full = bars;               // [S]
  uint64_t* empty = bars + S;          // [S]
  uint64_t* acc_full = bars + 2 * S;                // [kNumFree]
  uint64_t* acc_empty = acc_full + C::kNumFree;     // [kNumFree]
  uint64_t* drain = acc_empty + C::kNumFree;        // [1]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
  float* out_stage = reinterpret_cast<float*>(smem + S * C::kStageBytes + 512);  // STORE: [kEpiWarps][32][kOutPitch]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pair: rank 0 (the leader) issues the MMAs and owns the barriers both
  // CTAs' copies complete on and both CTAs' epilogues release; the pair walks
  // the units together (unit stride = number of pairs).
  const uint32_t rank = C::kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int64_t first_unit = C::kPair ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t unit_stride = C::kPair ? (gridDim.x >> 1) : gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::kNumFree; ++b) mbar_init(&acc_full[b], 1);
    // pair: one arrival per epilogue warp of both CTAs; otherwise every epilogue thread
    for (int b = 0; b < C::kNumFree; ++b) mbar_init(&acc_empty[b], C::kPair ? 2 * C::kEpiWarps : C::kEpiWarps * 32);
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_a0);
    tma_prefetch_desc(&tm_b0);
    if (MODE != kModeCE) {
      tma_prefetch_desc(&tm_a1);
      tma_prefetch_desc(&tm_b1);
    }
  }
  if (warp == 1) {
    if constexpr (C::kPair) {
      tmem_alloc_pair(s_tmem, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(s_tmem, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (C::kPair)
    cluster_sync();  // both CTAs' barriers initialised before any remote arrival or copy
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0, last_parity = 0;  // per-stage bit masks for the drain
      bool ok = true;
      for (int64_t u = first_unit; u < p.units && ok; u += unit_stride) {
        const UnitCoord c = decode_unit(p, u, MODE);
        const int kb_lo = store_mode<MODE>() ? c.head * p.kb_per : 0;
        const int kb_hi = store_mode<MODE>() ? min(p.k_blocks, kb_lo + p.kb_per) : p.k_blocks;
        for (int h = 0; h < C::kHeadsPerUnit && ok; ++h) {
          const int head = (MODE == kModeLSE) ? c.head : h;
          const CUtensorMap* ta = head ? &tm_a1 : &tm_a0;
          const CUtensorMap* tb = head ? &tm_b1 : &tm_b0;
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            // pair: the leader's commits free the stage in both CTAs
            const bool freed = C::kPair ? mbar_wait_cluster(&empty[stage], phase ^ 1u, p.timeout_ns, p.status)
                                        : mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, p.status);
            if (!freed) { ok = false; break; }
            uint8_t* sa = tiles + stage * C::kStageBytes;
            uint8_t* sb = sa + C::kABytes;
            if constexpr (C::kPair) {
              // both CTAs' copies complete on the leader's barrier, which expects them all
              if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
              const uint32_t fb = mapa_shared(&full[stage], 0);
              const int32_t arow = c.mt * C::kRowsM + static_cast<int32_t>(rank) * kBM;   // this CTA's A rows
              const int32_t brow = c.nt * BN + static_cast<int32_t>(rank) * C::kBRows;    // and B rows
              if (a_mn<MODE>()) {
                if (p.mn3d & 1u) {
                  tma_load_3d_pair(sa, ta, 0, kb * kBK, arow / kMnBox, fb);
                } else {
#pragma unroll
                  for (int j = 0; j < kBM / kMnBox; ++j)
                    tma_load_2d_pair(sa + j * kMnBoxBytes, ta, arow + j * kMnBox, kb * kBK, fb);
                }
              } else {
                tma_load_2d_pair(sa, ta, kb * kBK, arow, fb);
              }
              if (b_mn<MODE>()) {
                if (p.mn3d & 2u) {
                  tma_load_3d_pair(sb, tb, 0, kb * kBK, brow / kMnBox, fb);
                } else {
#pragma unroll
                  for (int j = 0; j < C::kBRows / kMnBox; ++j)
                    tma_load_2d_pair(sb + j * kMnBoxBytes, tb, brow + j * kMnBox, kb * kBK, fb);
                }
              } else {
                tma_load_2d_pair(sb, tb, kb * kBK, brow, fb);
              }
              filled |= 1u << stage;
              last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
              if (++stage == S) { stage = 0; phase ^= 1u; }
              continue;
            }
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
            // K-major operand: one box of 64 (K) x rows.  MN-major operand: boxes of
            // 64 (MN) x 64 (K), one per 64 rows of the tile, kMnBoxBytes apart --
            // as one 3-D copy when the map is 3-D, else one 2-D copy per box.
            if (a_mn<MODE>()) {
              if (p.mn3d & 1u) {
                tma_load_3d(sa, ta, 0, kb * kBK, c.mt * (kBM / kMnBox), &full[stage]);
              } else {
#pragma unroll
                for (int j = 0; j < kBM / kMnBox; ++j)
                  tma_load_2d(sa + j * kMnBoxBytes, ta, c.mt * kBM + j * kMnBox, kb * kBK, &full[stage]);
              }
            } else {
              tma_load_2d(sa, ta, kb * kBK, c.mt * kBM, &full[stage]);
            }
            if (b_mn<MODE>()) {
              if (p.mn3d & 2u) {
                tma_load_3d(sb, tb, 0, kb * kBK, c.nt * (BN / kMnBox), &full[stage]);
              } else {
#pragma unroll
                for (int j = 0; j < BN / kMnBox; ++j)
                  tma_load_2d(sb + j * kMnBoxBytes, tb, c.nt * BN + j * kMnBox, kb * kBK, &full[stage]);
              }
            } else {
              tma_load_2d(sb, tb, kb * kBK, c.nt * BN, &full[stage]);
            }
            filled |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
      }
      // Never leave with copies in flight: wait for the last fill of each stage
      // (pair: the leader's barriers count both CTAs' copies; the other CTA is
      // held by the closing cluster barrier until the leader has waited).
      for (int s = 0; s < S; ++s)
        if (filled & (1u << s)) {
          if constexpr (C::kPair) {
            if (leader) mbar_wait_cluster(&full[s], (last_parity >> s) & 1u, p.timeout_ns, p.status);
          } else {
            mbar_wait(&full[s], (last_parity >> s) & 1u, p.timeout_ns, p.status);
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(tiles);
      for (int64_t u = first_unit; u < p.units && ok; u += unit_stride) {
        const int kb_lo = store_mode<MODE>() ? decode_unit(p, u, MODE).head * p.kb_per : 0;
        const int kb_hi = store_mode<MODE>() ? min(p.k_blocks, kb_lo + p.kb_per) : p.k_blocks;
        if constexpr (!two_head<MODE>()) {
          const bool freed = C::kPair ? mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, p.status)
                                      : mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, p.status);
          if (!freed) break;
          tc_fence_after();
        }
        for (int h = 0; h < C::kHeadsPerUnit && ok; ++h) {
          if constexpr (two_head<MODE>()) {  // this head's columns released by the previous unit's epilogue
            if (!mbar_wait(&acc_empty[h], acc_phase ^ 1u, p.timeout_ns, p.status)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols + h * BN);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            const bool landed = C::kPair ? mbar_wait_cluster(&full[stage], phase, p.timeout_ns, p.status)
                                         : mbar_wait(&full[stage], phase, p.timeout_ns, p.status);
            if (!landed) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = a0 + stage * C::kStageBytes;
            // K step of 16: +32 bytes inside the swizzle row (K-major), +16 rows (MN-major)
            const uint64_t da = a_mn<MODE>() ? smem_desc_sw128_mn(sa) : smem_desc_sw128(sa);
            const uint64_t db = b_mn<MODE>() ? smem_desc_sw128_mn(sa + C::kABytes) : smem_desc_sw128(sa + C::kABytes);
            constexpr uint64_t kStepA = a_mn<MODE>() ? (16 * 128) >> 4 : 32 >> 4;
            constexpr uint64_t kStepB = b_mn<MODE>() ? (16 * 128) >> 4 : 32 >> 4;
            if constexpr (C::kPair) {
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                tc_mma_bf16_pair(d_tmem, da + kStepA * k, db + kStepB * k, C::kIdesc,
                                 (kb != kb_lo || k != 0) ? 1u : 0u);
              tc_commit_pair_mc(&empty[stage], 0x3);  // frees the stage in both CTAs
            } else {
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                tc_mma_bf16(d_tmem, da + kStepA * k, db + kStepB * k, C::kIdesc, (kb != kb_lo || k != 0) ? 1u : 0u);
              tc_commit(&empty[stage]);
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
          if constexpr (two_head<MODE>())
            if (ok) tc_commit(&acc_full[h]);  // this head's accumulator is complete
        }
        if (!ok) break;
        if constexpr (C::kPair)
          tc_commit_pair_mc(&acc_full[acc], 0x3);  // both CTAs' epilogues
        else if constexpr (!two_head<MODE>())
          tc_commit(&acc_full[acc]);
        if (++acc == C::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      if constexpr (C::kPair)
        tc_commit_pair_mc(drain, 0x1);
      else
        tc_commit(drain);
      mbar_wait(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                  // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;            // which column slice (kColSplit slices)
    constexpr int kCols = BN / C::kColSplit;    // columns of each head this warp reads
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    const float beta = p.beta, omb = 1.f - p.beta, it = p.inv_tau, it2 = p.inv_tau * kLog2e;
    for (int64_t u = first_unit; u < p.units; u += unit_stride) {
      const UnitCoord c = decode_unit(p, u, MODE);
      const int64_t row0 = static_cast<int64_t>(c.mt) * C::kRowsM + rank * kBM + quad * 32;  // this warp's rows
      const int64_t row = row0 + lane;
      const bool row_ok = row < p.T;
      const int64_t n0 = static_cast<int64_t>(c.nt) * BN + half * kCols;
      int64_t tgt = -1;
      float ls = 0.f, lt = 0.f;
      if ((MODE == kModeCE || MODE == kModeDZ) && row_ok) {
        tgt = __ldg(p.target + row);
        if (MODE == kModeCE) tgt = tgt >= p.v0 ? tgt - p.v0 : -1;  // column within this W (shard)
      }
      float gdz = 0.f;
      if (MODE == kModeDZ && row_ok) {
        ls = __ldg(p.lse + row);
        gdz = p.row_w ? p.gscale * __ldg(p.row_w + row) : p.gscale;
      }
      if (two_head<MODE>() && row_ok) {
        ls = __ldg(p.lse + row);
        lt = __ldg(p.lse + p.T + row);
      }
      const float ls2 = ls * kLog2e, lt2 = lt * kLog2e;  // log-sum-exps in base 2
      float krow = 0.f, gj = 0.f;
      if (MODE == kModeDZJ && row_ok) {
        krow = __ldg(p.kl + row);
        const bool kept = !p.keep || __ldg(p.keep + row);
        gj = kept ? p.gscale * __ldg(p.inv_count) * beta : 0.f;
      }
      // tcgen05.ld is warp-collective: the whole warp proceeds or gives up together
      const bool ok = __all_sync(0xFFFFFFFFu, C::kPair ? mbar_wait_cluster(&acc_full[acc], acc_phase, p.timeout_ns, p.status)
                                                       : mbar_wait(&acc_full[acc], acc_phase, p.timeout_ns, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + lane_addr + static_cast<uint32_t>(acc * C::kAccCols + half * kCols);
      MS st = ms_empty();
      float zt = 0.f;
      bool has_t = false;
      float jsd = 0.f, kacc = 0.f;
      if constexpr (two_head<MODE>()) {
        const bool walked = two_head_walk<kCols / 16>(
            tbase, BN, &acc_full[1], acc_phase, &acc_empty[0], &acc_empty[1], p.timeout_ns, p.status,
            [&](int cc, const uint32_t(&rs)[16], const uint32_t(&rt)[16]) {
          const int64_t col0 = n0 + cc * 16;
          if constexpr (MODE == kModeJSD) {
            if (col0 + 16 <= p.V) {
#if LMHO_JSD_PACKED
              const uint64_t i2 = f32x2(it2, it2), ns = f32x2(-ls2, -ls2), nt = f32x2(-lt2, -lt2);
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                jsd_term2_x2(jsd, f32x2(__uint_as_float(rs[j]), __uint_as_float(rs[j + 1])),
                             f32x2(__uint_as_float(rt[j]), __uint_as_float(rt[j + 1])), i2, ns, nt, beta, omb);
#else
#pragma unroll
              for (int j = 0; j < 16; ++j)
                jsd += jsd_term2(fmaf(__uint_as_float(rs[j]), it2, -ls2), fmaf(__uint_as_float(rt[j]), it2, -lt2),
                                 beta, omb);
#endif
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (col0 + j < p.V)
                  jsd += jsd_term2(fmaf(__uint_as_float(rs[j]), it2, -ls2),
                                   fmaf(__uint_as_float(rt[j]), it2, -lt2), beta, omb);
            }
          } else if constexpr (MODE == kModeJSDK) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (col0 + j < p.V) {
                float t, P, lplm2;
                jsd_term2_student(fmaf(__uint_as_float(rs[j]), it2, -ls2), fmaf(__uint_as_float(rt[j]), it2, -lt2),
                                  beta, omb, t, P, lplm2);
                jsd += t;
                kacc = fmaf(P, lplm2, kacc);   // KL(P || M) share in base 2, scaled by ln 2 when written
              }
            }
          } else {  // kModeDZJ: the student's dZ for this row and 16 columns
            // (written straight from registers: this epilogue is issue-bound, and a
            // shared-memory stage as in the DZ pass measured 5 % slower here)
            if (row_ok) {
              float g[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float P, lplm;
                jsd_student(fmaf(__uint_as_float(rs[j]), it, -ls), fmaf(__uint_as_float(rt[j]), it, -lt), beta,
                            omb, &P, &lplm);
                g[j] = (col0 + j < p.V) ? gj * P * (lplm - krow) : 0.f;
              }
              uint4* dst = reinterpret_cast<uint4*>(p.dz + row * p.ld_dz + col0);
#pragma unroll
              for (int k = 0; k < 2; ++k)
                dst[k] = make_uint4(pack_bf16x2(g[8 * k], g[8 * k + 1]), pack_bf16x2(g[8 * k + 2], g[8 * k + 3]),
                                    pack_bf16x2(g[8 * k + 4], g[8 * k + 5]), pack_bf16x2(g[8 * k + 6], g[8 * k + 7]));
            }
          }
        });
        if (!walked) break;
      } else {
#pragma unroll 1
        for (int cc = 0; cc < kCols / 32; ++cc) {
          const int64_t col0 = n0 + cc * 32;
          if (MODE == kModeDZ) {
            float v[32];
            tmem_ld32_sync(tbase + cc * 32, v);
            // a vocabulary shard: the target is global, its column here is tgt - v0
            const bool bad = tgt < 0 || tgt >= (p.v_total ? p.v_total : p.V);
            const int64_t tl = bad ? -1 : tgt - p.v0;
            const float g = gdz, nl = -ls * kLog2e;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t col = col0 + j;
              float d = col < p.V ? g * ex2_approx(fmaf(v[j], kLog2e, nl)) : 0.f;
              if (col == tl) d -= g;
              v[j] = bad ? __int_as_float(0x7FC00000) : d;
            }
            // Each lane's 64-byte dZ row segment (32 bf16; ld_dz is a multiple of the
            // tile width) goes through shared memory: 16-byte chunk k of row r sits
            // at r * 64 + (k ^ ((r >> 1) & 3)) * 16, so both the row-per-lane writes
            // and the 4-lanes-per-row reads are free of bank conflicts; the global
            // writes then cover 8 rows x 64 contiguous bytes per instruction.
            uint8_t* sw = reinterpret_cast<uint8_t*>(out_stage) + (warp - 2) * 32 * 64;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<uint4*>(sw + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                             pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 8 * i + (lane >> 2), k = lane & 3;
              const uint4 val = *reinterpret_cast<const uint4*>(sw + r * 64 + ((k ^ ((r >> 1) & 3)) << 4));
              if (row0 + r < p.T) *reinterpret_cast<uint4*>(p.dz + (row0 + r) * p.ld_dz + col0 + 8 * k) = val;
            }
            __syncwarp();
          } else if (store_mode<MODE>()) {
            // Lane = row: stage the warp's 32 rows x 32 columns in shared memory,
            // then write them back 4 rows x 128 contiguous bytes per instruction
            // (8 lanes per row) instead of 32 rows x 16 bytes.
            float v[32];
            tmem_ld32_sync(tbase + cc * 32, v);
            float* sw = out_stage + (warp - 2) * 32 * C::kOutPitch;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(sw + lane * C::kOutPitch + 4 * k) =
                  make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            __syncwarp();
            const int c4 = (lane & 7) * 4;
            float* obase = p.out + c.head * p.split_stride + col0 + c4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + (lane >> 3);
              const float4 val = *reinterpret_cast<const float4*>(sw + r * C::kOutPitch + c4);
              if (row0 + r < p.T) {
                float* dst = obase + (row0 + r) * p.ld_out;
                if (col0 + c4 + 4 <= p.V) {
                  *reinterpret_cast<float4*>(dst) = val;
                } else {
                  if (col0 + c4 < p.V) dst[0] = val.x;
                  if (col0 + c4 + 1 < p.V) dst[1] = val.y;
                  if (col0 + c4 + 2 < p.V) dst[2] = val.z;
                }
              }
            }
            __syncwarp();
          } else {
            float v[32];
            tmem_ld32_sync(tbase + cc * 32, v);
            if (MODE == kModeLSE) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] *= p.inv_tau;
            }
            if (col0 + 32 > p.V) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= p.V) v[j] = -INFINITY;
            }
            if (MODE == kModeCE) {
              const int64_t off = tgt - col0;
              if (off >= 0 && off < 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j == off) zt = v[j];
                has_t = true;
              }
            }
#if LMHO_FOLD_PACKED
            ms_fold_packed<32>(st, v);
#else
            ms_fold<32>(st, v);
#endif
          }
        }
      }
      // accumulator fully read: hand it back to the MMA warp (two-head: done per head by the walk)
      if constexpr (C::kPair) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(&acc_empty[acc], 0));
      } else if constexpr (!two_head<MODE>()) {
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
      }
      if (++acc == C::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      if (row_ok && (MODE == kModeCE || MODE == kModeLSE || MODE == kModeJSD || MODE == kModeJSDK)) {
        // partial slot of this (vocab tile, column slice)
        const int64_t slot = static_cast<int64_t>(c.nt) * C::kColSplit + half;
        if (MODE == kModeJSD || MODE == kModeJSDK) {
          p.part0[slot * p.T + row] = -kLn2 * jsd;
          if (MODE == kModeJSDK) p.part1[slot * p.T + row] = kLn2 * kacc;
        } else {
          const int64_t idx = (static_cast<int64_t>(c.head) * p.num_n * C::kColSplit + slot) * p.T + row;
          p.part0[idx] = st.m;
          p.part1[idx] = st.s;
          if (MODE == kModeCE && has_t) p.part2[slot * p.T + row] = zt;
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (C::kPair)
    cluster_sync();  // neither CTA leaves while the pair's MMAs, copies or arrivals may touch it
  else
    __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (C::kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- finalisers
constexpr int kFinRows = 32;   // rows per block (one per lane)
constexpr int kFinSplit = 16;  // warps per block, each merging a slice of the vocab tiles

// Merge (m, s) partials [num_n][T] of each row, in vocab-tile order, into
// its log-sum-exp.  Warp w handles tiles [w*cnt, (w+1)*cnt); the kFinSplit results
// merge in warp order.
__device__ __forceinline__ MS merge_ms_row(const float* pm, const float* ps, int64_t T, int num_n, int64_t row,
                                           MS* s_tmp) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int cnt = (num_n + kFinSplit - 1) / kFinSplit;
  const int n_lo = min(num_n, w * cnt), n_hi = min(num_n, n_lo + cnt);
  MS a = ms_empty();
  if (row < T) {
#pragma unroll 4
    for (int n = n_lo; n < n_hi; ++n) {
      const int64_t i = static_cast<int64_t>(n) * T + row;
      a = ms_merge(a, MS{__ldcg(pm + i), __ldcg(ps + i)});
    }
  }
  s_tmp[w * 32 + l] = a;
  __syncthreads();
  MS tot = s_tmp[l];
  for (int k = 1; k < kFinSplit; ++k) tot = ms_merge(tot, s_tmp[k * 32 + l]);
  __syncthreads();
  return tot;  // meaningful in warp 0
}
__device__ __forceinline__ float merge_lse_row(const float* pm, const float* ps, int64_t T, int num_n,
                                               int64_t row, MS* s_tmp) {
  const MS tot = merge_ms_row(pm, ps, T, num_n, row, s_tmp);
  return tot.m + logf(tot.s);
}

__global__ void __launch_bounds__(kFinRows * kFinSplit)
    flce_finalize(const float* pm, const float* ps, const float* pz, const int64_t* target, int64_t T,
                  int64_t V, int num_n, float* row_out, float* loss, Ctrl* ctrl, float* lse_out) {
  __shared__ MS s_tmp[kFinRows * kFinSplit];
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kFinRows + (threadIdx.x & 31);
  const float lse = merge_lse_row(pm, ps, T, num_n, row, s_tmp);
  if (threadIdx.x < 32 && row < T) {
    const int64_t t = __ldg(target + row);
    float zt = __int_as_float(0x7FC00000);
    if (t >= 0 && t < V) zt = __ldcg(pz + (t / kBN_CE) * T + row);
    row_out[row] = lse - zt;
    if (lse_out) lse_out[row] = lse;
  }
  mean_tail(row_out, T, loss, ctrl, gridDim.x);
}

// One vocabulary shard of the fused linear + CE (W = the global rows [v0, v0 + V)):
// each token's (max, sum of exp) over the shard, merged over its vocab tiles
// as in flce_finalize, and its target logit when the (global) target is in
// the shard, else -inf; written as part [3][T] (m, s, z).
__global__ void __launch_bounds__(kFinRows * kFinSplit)
    flce_partials_finalize(const float* pm, const float* ps, const float* pz, const int64_t* target, int64_t T,
                           int64_t V, int64_t v0, int num_n, float* part) {
  __shared__ MS s_tmp[kFinRows * kFinSplit];
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kFinRows + (threadIdx.x & 31);
  const MS tot = merge_ms_row(pm, ps, T, num_n, row, s_tmp);
  if (threadIdx.x < 32 && row < T) {
    const int64_t t = __ldg(target + row);
    float zt = -INFINITY;
    if (t >= v0 && t - v0 < V) zt = __ldcg(pz + ((t - v0) / kBN_CE) * T + row);
    part[row] = tot.m;
    part[T + row] = tot.s;
    part[2 * T + row] = zt;
  }
}

__global__ void __launch_bounds__(kFinRows * kFinSplit)
    lse_finalize(const float* pm, const float* ps, int64_t T, int num_n, float* lse_out) {
  __shared__ MS s_tmp[kFinRows * kFinSplit];
  const int head = blockIdx.y;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kFinRows + (threadIdx.x & 31);
  const int64_t hoff = static_cast<int64_t>(head) * num_n * T;
  const float lse = merge_lse_row(pm + hoff, ps + hoff, T, num_n, row, s_tmp);
  if (threadIdx.x < 32 && row < T) lse_out[head * T + row] = lse;
}

__global__ void __launch_bounds__(kFinRows * kFinSplit)
    jsd_finalize(const float* pj, int64_t T, int num_n, const uint8_t* keep, float* row_out, float* loss, Ctrl* ctrl,
                 const float* pk = nullptr, float* kl_out = nullptr, float* inv_count_out = nullptr) {
  __shared__ float s_tmp[kFinRows * kFinSplit];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kFinRows + l;
  const int cnt = (num_n + kFinSplit - 1) / kFinSplit;
  const int n_lo = min(num_n, w * cnt), n_hi = min(num_n, n_lo + cnt);
  KSum a;   // compensated fp32: the partial sums are added in tile order
  if (row < T) {
#pragma unroll 4
    for (int n = n_lo; n < n_hi; ++n) a.add(__ldcg(pj + static_cast<int64_t>(n) * T + row));
  }
  s_tmp[w * 32 + l] = a.s - a.c;
  __syncthreads();
  if (w == 0 && row < T) {
    KSum tot;
    for (int k = 0; k < kFinSplit; ++k) tot.add(s_tmp[k * 32 + l]);
    row_out[row] = (keep && !__ldg(keep + row)) ? 0.f : tot.s - tot.c;
  }
  if (pk) {  // the same fixed-order sum of the KL(P || M) partials
    __syncthreads();
    KSum b;
    if (row < T) {
#pragma unroll 4
      for (int n = n_lo; n < n_hi; ++n) b.add(__ldcg(pk + static_cast<int64_t>(n) * T + row));
    }
    s_tmp[w * 32 + l] = b.s - b.c;
    __syncthreads();
    if (w == 0 && row < T) {
      KSum tot;
      for (int k = 0; k < kFinSplit; ++k) tot.add(s_tmp[k * 32 + l]);
      kl_out[row] = tot.s - tot.c;
    }
  }
  if (loss) mean_tail(row_out, T, loss, ctrl, gridDim.x, keep, inv_count_out);  // null: per-row sums only
}

// CPO from the per-token CE losses rows [B * S] (published objective, Xu et
// al. 2024; page "Fused linear + CPO loss" names it): sequence b < B/2 is the
// chosen answer of pair b, sequence b + B/2 its rejected answer.  One block of
// 256 threads per sequence: thread j sums tokens j, j + 256, ... (compensated),
// then a fixed butterfly and the 8 warp sums in order give lp_b = -sum.  The
// last block to finish (atomic ticket) combines the pairs in order:
//   d_k = lp_k - lp_{k+Bc},  loss = alpha (sum_{b<Bc} -lp_b) / (Bc S)
//                                  + (1/Bc) sum_k softplus(-beta d_k),
// keeping sig_k = sigmoid(-beta d_k); with row_w set it then writes
// d loss / d l_i: alpha/(Bc S) + (beta/Bc) sig_k for a chosen token of pair k,
// -(beta/Bc) sig_k for a rejected one; and leaves the ticket at 0.
__global__ void __launch_bounds__(256)
    cpo_finalize(const float* rows, int64_t B, int64_t S, float beta, float alpha, float* lp, float* sig, float* loss,
                 float* logps, float* row_w, Ctrl* ctrl) {
  __shared__ float s_warp[8];
  __shared__ uint32_t s_last;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int64_t b = blockIdx.x;
  KSum a;
  for (int64_t s = threadIdx.x; s < S; s += 256) a.add(__ldcg(rows + b * S + s));
  float v = a.s - a.c;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (l == 0) s_warp[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += s_warp[k];
    lp[b] = -t;
    if (logps) logps[b] = -t;
    __threadfence();
    s_last = atomicAdd(&ctrl->ticket, 1u) == gridDim.x - 1 ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t Bc = B / 2;
  if (threadIdx.x == 0) {
    KSum pref, nll;
    for (int64_t k = 0; k < Bc; ++k) {
      const float lc = __ldcg(lp + k);
      const float u = -beta * (lc - __ldcg(lp + k + Bc));
      const float e = expf(-fabsf(u));
      pref.add(fmaxf(u, 0.f) + log1pf(e));
      sig[k] = u >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
      nll.add(-lc);
    }
    *loss = alpha * (nll.s - nll.c) / (static_cast<float>(Bc) * static_cast<float>(S)) +
            (pref.s - pref.c) / static_cast<float>(Bc);
    ctrl->ticket = 0u;
    __threadfence();
  }
  if (!row_w) return;
  __syncthreads();
  const float aw = alpha / (static_cast<float>(Bc) * static_cast<float>(S)), bw = beta / static_cast<float>(Bc);
  for (int64_t i = threadIdx.x; i < B * S; i += blockDim.x) {
    const int64_t q = i / S;
    row_w[i] = q < Bc ? fmaf(bw, sig[q], aw) : -bw * sig[q - Bc];
  }
}

// out[i] = sum over s = 0 .. splits-1, in that order, of part[s * n + i]: the
// K slices of a split gradient GEMM folded into the caller's buffer.  n % 4 == 0
// and both buffers 16-byte aligned (checked by the caller).
__global__ void __launch_bounds__(256)
    split_sum(const float* __restrict__ part, int splits, int64_t n, float* __restrict__ out) {
  const int64_t n4 = n >> 2;
  const float4* p4 = reinterpret_cast<const float4*>(part);
  float4* o4 = reinterpret_cast<float4*>(out);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = __ldcs(p4 + i);
    for (int k = 1; k < splits; ++k) {
      const float4 b = __ldcs(p4 + k * n4 + i);
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    o4[i] = a;
  }
}

__global__ void wait_selftest_kernel(Ctrl* ctrl, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    // Nothing ever arrives on `bar`: the bounded wait must give up and report.
    mbar_wait(&bar, 0, timeout_ns, &ctrl->status);
  }
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                        const CUtensorMap& b1, const Params& p, const FusedLaunch& L) {
  using C = ModeCfg<MODE>;
  static std::atomic<bool> limit_set[kMaxDevices];
  if (const cudaError_t e = ensure_smem_limit(fused_gemm_kernel<MODE>, C::kSmemBytes, limit_set); e != cudaSuccess)
    return e;
  if constexpr (C::kPair) {
    // clusters of 2 CTAs (one per SM): as many pairs as can be resident at once
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    // resident pairs per device, queried once (0 = not yet; atomic: calls may
    // come from several host threads, and racing first queries agree)
    static std::atomic<int> pairs_max[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    int cap = dev < kMaxDevices ? pairs_max[dev].load(std::memory_order_relaxed) : 0;
    if (cap == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(2 * (L.num_sms / 2)));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fused_gemm_kernel<MODE>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = L.num_sms / 2;
      }
      cap = n < L.num_sms / 2 ? n : L.num_sms / 2;
      if (cap < 1) cap = 1;
      if (dev < kMaxDevices) pairs_max[dev].store(cap, std::memory_order_relaxed);
    }
    const int64_t pairs = p.units < cap ? p.units : cap;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    return cudaLaunchKernelEx(&cfg, fused_gemm_kernel<MODE>, a0, b0, a1, b1, p);
  } else {
    const int64_t grid = p.units < L.num_sms ? p.units : L.num_sms;
    fused_gemm_kernel<MODE><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, L.stream>>>(a0, b0, a1, b1,
                                                                                                   p);
    return cudaGetLastError();
  }
}

// Tile grid of a MODE's units: token tiles of ModeCfg<MODE>::kRowsM rows (a
// pair's tile is two of the geometry's kBM-row tiles), and a raster group
// spanning the same tokens as the geometry's.
template <int MODE>
Params base_params(const FusedGeometry& g, const FusedLaunch& L, Ctrl* ctrl) {
  constexpr int rows = ModeCfg<MODE>::kRowsM;
  Params p{};
  p.T = g.T;
  p.V = g.V;
  p.num_m = static_cast<int32_t>((g.T + rows - 1) / rows);
  p.num_n = static_cast<int32_t>(g.num_n);
  const int gm = static_cast<int>(static_cast<int64_t>(g.group_m) * kBM / rows);
  p.group_m = gm > 1 ? (gm < p.num_m ? gm : p.num_m) : 1;
  p.k_blocks = static_cast<int32_t>((g.H + kBK - 1) / kBK);
  p.timeout_ns = L.timeout_ns;
  p.status = &ctrl->status;
  p.inv_tau = 1.f;
  return p;
}

}  // namespace

cudaError_t launch_flce(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target,
                        const FusedGeometry& g, float* loss, const FusedWs& ws, const FusedLaunch& L) {
  Params p = base_params<kModeCE>(g, L, ws.ctrl);
  p.units = static_cast<int64_t>(p.num_m) * p.num_n;
  p.target = target;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.part2 = ws.part2;
  launch_mark(0, L.stream);
  cudaError_t e = launch_gemm<kModeCE>(tm_x, tm_w, tm_x, tm_w, p, L);
  if (e != cudaSuccess) return e;
  launch_mark(1, L.stream);
  const unsigned blocks = static_cast<unsigned>((g.T + kFinRows - 1) / kFinRows);
  flce_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, ws.part2, target, g.T, g.V,
                                                               static_cast<int>(g.num_n), ws.row_out, loss, ws.ctrl,
                                                               nullptr);
  launch_mark(2, L.stream);
  return cudaGetLastError();
}

cudaError_t launch_fljsd(const CUtensorMap& tm_xs, const CUtensorMap& tm_ws256, const CUtensorMap& tm_xt,
                         const CUtensorMap& tm_wt256, const CUtensorMap& tm_wsj, const CUtensorMap& tm_wtj,
                         const FusedGeometry& g_lse, const FusedGeometry& g_jsd, float beta, float inv_tau,
                         const uint8_t* keep, float* loss, const FusedWs& ws, const FusedLaunch& L) {
  // pass 1: log-sum-exp of both heads
  Params p = base_params<kModeLSE>(g_lse, L, ws.ctrl);
  p.units = 2 * static_cast<int64_t>(p.num_m) * p.num_n;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.inv_tau = inv_tau;
  launch_mark(0, L.stream);
  cudaError_t e = launch_gemm<kModeLSE>(tm_xs, tm_ws256, tm_xt, tm_wt256, p, L);
  if (e != cudaSuccess) return e;
  launch_mark(1, L.stream);
  dim3 fb(static_cast<unsigned>((g_lse.T + kFinRows - 1) / kFinRows), 2);
  lse_finalize<<<fb, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, g_lse.T, static_cast<int>(g_lse.num_n),
                                                          ws.lse);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_mark(2, L.stream);
  // pass 2: recompute both heads' tiles, accumulate the divergence
  Params q = base_params<kModeJSD>(g_jsd, L, ws.ctrl);
  q.units = static_cast<int64_t>(q.num_m) * q.num_n;
  q.part0 = ws.part0;
  q.lse = ws.lse;
  q.beta = beta;
  q.inv_tau = inv_tau;
  e = launch_gemm<kModeJSD>(tm_xs, tm_wsj, tm_xt, tm_wtj, q, L);
  if (e != cudaSuccess) return e;
  launch_mark(3, L.stream);
  const unsigned blocks = static_cast<unsigned>((g_jsd.T + kFinRows - 1) / kFinRows);
  jsd_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(
      ws.part0, g_jsd.T, static_cast<int>(g_jsd.num_n * ModeCfg<kModeJSD>::kColSplit), keep, ws.row_out, loss,
      ws.ctrl);
  launch_mark(4, L.stream);
  return cudaGetLastError();
}

cudaError_t launch_flce_partials(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target, int64_t v0,
                                 const FusedGeometry& g, float* partials, const FusedWs& ws, const FusedLaunch& L) {
  Params p = base_params<kModeCE>(g, L, ws.ctrl);
  p.units = static_cast<int64_t>(p.num_m) * p.num_n;
  p.target = target;
  p.v0 = v0;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.part2 = ws.part2;
  launch_mark(0, L.stream);
  cudaError_t e = launch_gemm<kModeCE>(tm_x, tm_w, tm_x, tm_w, p, L);
  if (e != cudaSuccess) return e;
  launch_mark(1, L.stream);
  const unsigned blocks = static_cast<unsigned>((g.T + kFinRows - 1) / kFinRows);
  flce_partials_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(
      ws.part0, ws.part1, ws.part2, target, g.T, g.V, v0, static_cast<int>(g.num_n), partials);
  launch_mark(2, L.stream);
  return cudaGetLastError();
}

cudaError_t launch_fljsd_lse_shard(const CUtensorMap& tm_xs, const CUtensorMap& tm_ws256, const CUtensorMap& tm_xt,
                                   const CUtensorMap& tm_wt256, const FusedGeometry& g_lse, float inv_tau,
                                   float* lse_local, const FusedWs& ws, const FusedLaunch& L) {
  Params p = base_params<kModeLSE>(g_lse, L, ws.ctrl);
  p.units = 2 * static_cast<int64_t>(p.num_m) * p.num_n;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.inv_tau = inv_tau;
  launch_mark(0, L.stream);
  cudaError_t e = launch_gemm<kModeLSE>(tm_xs, tm_ws256, tm_xt, tm_wt256, p, L);
  if (e != cudaSuccess) return e;
  launch_mark(1, L.stream);
  dim3 fb(static_cast<unsigned>((g_lse.T + kFinRows - 1) / kFinRows), 2);
  lse_finalize<<<fb, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, g_lse.T, static_cast<int>(g_lse.num_n),
                                                          lse_local);
  launch_mark(2, L.stream);
  return cudaGetLastError();
}

cudaError_t launch_fljsd_terms_shard(const CUtensorMap& tm_xs, const CUtensorMap& tm_wsj, const CUtensorMap& tm_xt,
                                     const CUtensorMap& tm_wtj, const FusedGeometry& g_jsd, const float* lse,
                                     float beta, float inv_tau, float* terms, float* kl_local, const FusedWs& ws,
                                     const FusedLaunch& L) {
  launch_mark(0, L.stream);
  cudaError_t e;
  if (kl_local) {  // the backward's variant: also each token's share of KL(P || M); the same divergence bits
    Params q = base_params<kModeJSDK>(g_jsd, L, ws.ctrl);
    q.units = static_cast<int64_t>(q.num_m) * q.num_n;
    q.part0 = ws.part0;
    q.part1 = ws.part1;
    q.lse = lse;
    q.beta = beta;
    q.inv_tau = inv_tau;
    if ((e = launch_gemm<kModeJSDK>(tm_xs, tm_wsj, tm_xt, tm_wtj, q, L)) != cudaSuccess) return e;
  } else {
    Params q = base_params<kModeJSD>(g_jsd, L, ws.ctrl);
    q.units = static_cast<int64_t>(q.num_m) * q.num_n;
    q.part0 = ws.part0;
    q.lse = lse;
    q.beta = beta;
    q.inv_tau = inv_tau;
    if ((e = launch_gemm<kModeJSD>(tm_xs, tm_wsj, tm_xt, tm_wtj, q, L)) != cudaSuccess) return e;
  }
  launch_mark(1, L.stream);
  const unsigned blocks = static_cast<unsigned>((g_jsd.T + kFinRows - 1) / kFinRows);
  static_assert(ModeCfg<kModeJSD>::kColSplit == ModeCfg<kModeJSDK>::kColSplit, "one partial layout");
  jsd_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(
      ws.part0, g_jsd.T, static_cast<int>(g_jsd.num_n * ModeCfg<kModeJSD>::kColSplit), nullptr, terms, nullptr,
      ws.ctrl, kl_local ? ws.part1 : nullptr, kl_local);
  launch_mark(2, L.stream);
  return cudaGetLastError();
}

cudaError_t launch_cpo_combine(const float* rows, int64_t B, int64_t S, float beta, float alpha, float* loss,
                               float* logps, float* row_w, float* lp, float* sig, Ctrl* ctrl, cudaStream_t st) {
  launch_mark(0, st);
  cpo_finalize<<<static_cast<unsigned>(B), 256, 0, st>>>(rows, B, S, beta, alpha, lp, sig, loss, logps, row_w, ctrl);
  launch_mark(1, st);
  return cudaGetLastError();
}

cudaError_t launch_flce_cpo(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target,
                            const FusedGeometry& g, float* loss, const FusedWs& ws, const CpoArgs& c,
                            const FusedLaunch& L) {
  Params p = base_params<kModeCE>(g, L, ws.ctrl);
  p.units = static_cast<int64_t>(p.num_m) * p.num_n;
  p.target = target;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.part2 = ws.part2;
  launch_mark(0, L.stream);
  cudaError_t e = launch_gemm<kModeCE>(tm_x, tm_w, tm_x, tm_w, p, L);
  if (e != cudaSuccess) return e;
  launch_mark(1, L.stream);
  const unsigned blocks = static_cast<unsigned>((g.T + kFinRows - 1) / kFinRows);
  flce_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, ws.part2, target, g.T, g.V,
                                                               static_cast<int>(g.num_n), ws.row_out, c.mean, ws.ctrl,
                                                               nullptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cpo_finalize<<<static_cast<unsigned>(c.B), 256, 0, L.stream>>>(ws.row_out, c.B, c.S, c.beta, c.alpha, c.lp, c.sig,
                                                                 loss, c.logps, nullptr, ws.ctrl);
  launch_mark(2, L.stream);
  return cudaGetLastError();
}

int choose_k_split(int64_t tiles, int k_blocks, int num_sms) {
  if (tiles >= kSplitTiles || num_sms <= 0) return 1;
  auto fill = [&](int s) {  // share of the SM slots the last wave leaves busy
    const int64_t units = tiles * s;
    const int64_t waves = (units + num_sms - 1) / num_sms;
    return static_cast<double>(units) / static_cast<double>(waves * num_sms);
  };
  int best = 1;
  double best_fill = fill(1);
  for (int s = 2; s <= kMaxKSplit && k_blocks / s >= kMinSplitKBlocks; ++s) {
    const double f = fill(s);
    if (f > best_fill + 0.02) {  // each slice costs a partial write and read
      best = s;
      best_fill = f;
    }
  }
  return best;
}

size_t k_split_reserve_bytes(int64_t M, int64_t N) {
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN_CE - 1) / kBN_CE);
  return tiles < kSplitTiles ? static_cast<size_t>(kMaxKSplit) * 4 * static_cast<size_t>(M) * N : 0;
}

namespace {
// out [M, N] fp32 (row stride N) = A B with K = `K`, operands read through the
// tensor maps the MODE expects.  With fewer output tiles than kSplitTiles the
// K range is cut into slices written to `split_ws` and summed in slice order.
template <int MODE>
cudaError_t launch_store_gemm(const CUtensorMap& a, const CUtensorMap& b, int64_t M, int64_t N, int64_t K, float* out,
                              float* split_ws, int group_m, Ctrl* ctrl, const FusedLaunch& L) {
  FusedGeometry g{};
  g.T = M;
  g.V = N;
  g.H = K;
  g.num_m = (M + kBM - 1) / kBM;
  g.num_n = (N + kBN_CE - 1) / kBN_CE;
  g.group_m = static_cast<int>(g.num_m < group_m ? g.num_m : group_m);
  Params p = base_params<MODE>(g, L, ctrl);
  const int64_t tiles = static_cast<int64_t>(p.num_m) * p.num_n;
  // a pair's tile occupies two SMs: plan the split in one-SM tile slots
  const int64_t slots = ModeCfg<MODE>::kPair ? 2 * tiles : tiles;
  int splits = split_ws ? choose_k_split(slots, p.k_blocks, L.num_sms) : 1;
  p.kb_per = (p.k_blocks + splits - 1) / splits;
  splits = (p.k_blocks + p.kb_per - 1) / p.kb_per;  // no empty slice
  p.k_split = splits;
  p.units = tiles * splits;
  p.out = splits > 1 ? split_ws : out;
  p.ld_out = N;
  p.split_stride = M * N;
  // the MN-major maps were made 3-D exactly when their MN extent is whole chunks
  p.mn3d = (a_mn<MODE>() && mn_chunked(M) ? 1u : 0u) | (b_mn<MODE>() && mn_chunked(N) ? 2u : 0u);
  cudaError_t e = launch_gemm<MODE>(a, b, a, b, p, L);
  if (e != cudaSuccess || splits == 1) return e;
  const int64_t n4 = M * N / 4;
  const int64_t cap = static_cast<int64_t>(L.num_sms) * 8;
  const int64_t blocks = (n4 + 255) / 256 < cap ? (n4 + 255) / 256 : cap;
  split_sum<<<static_cast<unsigned>(blocks), 256, 0, L.stream>>>(split_ws, splits, M * N, out);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_flce_fwd_bwd(const FlceBwdMaps& m, const int64_t* target, const FusedGeometry& g, float grad_scale,
                                float* loss, float* dx, float* dW, const FusedWs& ws, const FlceBwdWs& bw,
                                const FusedLaunch& L, const CpoArgs* cpo) {
  cudaError_t e;
  launch_mark(0, L.stream);
  // forward: per-token loss, mean, and each row's log-sum-exp
  Params p = base_params<kModeCE>(g, L, ws.ctrl);
  p.units = static_cast<int64_t>(p.num_m) * p.num_n;
  p.target = target;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.part2 = ws.part2;
  if ((e = launch_gemm<kModeCE>(m.x, m.w, m.x, m.w, p, L)) != cudaSuccess) return e;
  const unsigned fblocks = static_cast<unsigned>((g.T + kFinRows - 1) / kFinRows);
  flce_finalize<<<fblocks, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, ws.part2, target, g.T, g.V,
                                                                static_cast<int>(g.num_n), ws.row_out,
                                                                cpo ? cpo->mean : loss, ws.ctrl, bw.lse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (cpo) {  // CPO: the loss and each token's weight d loss / d l_i
    cpo_finalize<<<static_cast<unsigned>(cpo->B), 256, 0, L.stream>>>(
        ws.row_out, cpo->B, cpo->S, cpo->beta, cpo->alpha, cpo->lp, cpo->sig, loss, cpo->logps, cpo->row_w, ws.ctrl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  launch_mark(1, L.stream);
  // recompute the logit tiles, write dZ
  Params q = base_params<kModeDZ>(g, L, ws.ctrl);
  q.units = static_cast<int64_t>(q.num_m) * q.num_n;
  q.target = target;
  q.lse = bw.lse;
  q.gscale = cpo ? grad_scale : grad_scale / static_cast<float>(g.T);
  q.row_w = cpo ? cpo->row_w : nullptr;
  q.dz = bw.dz;
  q.ld_dz = bw.ld_dz;
  if ((e = launch_gemm<kModeDZ>(m.x, m.w, m.x, m.w, q, L)) != cudaSuccess) return e;
  launch_mark(2, L.stream);
  // dx [T, H] = dZ [T, V] W [V, H]  (K = V; W read MN-major)
  if ((e = launch_store_gemm<kModeStore>(m.dz, m.w_mn, g.T, g.H, g.V, dx, bw.split, g.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(3, L.stream);
  // dW [V, H] = dZ^T [V, T] x [T, H]  (K = T; dZ and x read MN-major)
  if ((e = launch_store_gemm<kModeStoreT>(m.dz_mn, m.x_mn, g.V, g.H, g.T, dW, bw.split, g.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(4, L.stream);
  return cudaSuccess;
}

cudaError_t launch_flce_shard_bwd(const FlceBwdMaps& m, const int64_t* target, const float* partials,
                                  int64_t shards, int64_t v0, int64_t v_total, const FusedGeometry& g,
                                  float grad_scale, const float* row_w, float* dx, float* dW, const FusedWs& ws,
                                  const FlceBwdWs& bw, const FusedLaunch& L) {
  cudaError_t e;
  launch_mark(0, L.stream);
  // each token's global log-sum-exp from every shard's partials
  if ((e = launch_partials_lse(partials, shards, g.T, bw.lse, L.num_sms, L.stream)) != cudaSuccess) return e;
  // recompute the shard's logit tiles, write its dZ columns
  Params q = base_params<kModeDZ>(g, L, ws.ctrl);
  q.units = static_cast<int64_t>(q.num_m) * q.num_n;
  q.target = target;
  q.v0 = v0;
  q.v_total = v_total;
  q.lse = bw.lse;
  // the mean's weight 1/T on every row, or the caller's per-row weights (e.g. CPO's d loss / d l_i)
  q.gscale = row_w ? grad_scale : grad_scale / static_cast<float>(g.T);
  q.row_w = row_w;
  q.dz = bw.dz;
  q.ld_dz = bw.ld_dz;
  if ((e = launch_gemm<kModeDZ>(m.x, m.w, m.x, m.w, q, L)) != cudaSuccess) return e;
  launch_mark(1, L.stream);
  // this shard's share of dx [T, H] = dZ_shard W_local, and its rows of dW = dZ_shard^T x
  if ((e = launch_store_gemm<kModeStore>(m.dz, m.w_mn, g.T, g.H, g.V, dx, bw.split, g.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(2, L.stream);
  if ((e = launch_store_gemm<kModeStoreT>(m.dz_mn, m.x_mn, g.V, g.H, g.T, dW, bw.split, g.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(3, L.stream);
  return cudaSuccess;
}

cudaError_t launch_fljsd_fwd_bwd(const FljsdBwdMaps& m, const FusedGeometry& g_lse, const FusedGeometry& g_jsd,
                                 float beta, float inv_tau, const uint8_t* keep, float grad_scale, float* loss,
                                 float* dxs, float* dWs, const FusedWs& ws, const FlceBwdWs& bw, float* kl,
                                 float* inv_count, const FusedLaunch& L) {
  cudaError_t e;
  const int64_t T = g_lse.T, H = g_lse.H, V = g_lse.V;
  launch_mark(0, L.stream);
  // pass 1: log-sum-exp of both heads
  Params p = base_params<kModeLSE>(g_lse, L, ws.ctrl);
  p.units = 2 * static_cast<int64_t>(p.num_m) * p.num_n;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.inv_tau = inv_tau;
  if ((e = launch_gemm<kModeLSE>(m.xs, m.ws256, m.xt, m.wt256, p, L)) != cudaSuccess) return e;
  dim3 fb(static_cast<unsigned>((T + kFinRows - 1) / kFinRows), 2);
  lse_finalize<<<fb, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, T, static_cast<int>(g_lse.num_n), ws.lse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // pass 2: divergence and KL(P || M) of every row
  Params q = base_params<kModeJSDK>(g_jsd, L, ws.ctrl);
  q.units = static_cast<int64_t>(q.num_m) * q.num_n;
  q.part0 = ws.part0;
  q.part1 = ws.part1;
  q.lse = ws.lse;
  q.beta = beta;
  q.inv_tau = inv_tau;
  if ((e = launch_gemm<kModeJSDK>(m.xs, m.wsj, m.xt, m.wtj, q, L)) != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((T + kFinRows - 1) / kFinRows);
  const int nslots = static_cast<int>(g_jsd.num_n * ModeCfg<kModeJSDK>::kColSplit);
  jsd_finalize<<<blocks, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, T, nslots, keep, ws.row_out, loss, ws.ctrl,
                                                              ws.part1, kl, inv_count);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  launch_mark(1, L.stream);
  // pass 3: both heads again, the student's dZ
  Params r = base_params<kModeDZJ>(g_jsd, L, ws.ctrl);
  r.units = static_cast<int64_t>(r.num_m) * r.num_n;
  r.lse = ws.lse;
  r.beta = beta;
  r.inv_tau = inv_tau;
  r.gscale = grad_scale * inv_tau;
  r.kl = kl;
  r.keep = keep;
  r.inv_count = inv_count;
  r.dz = bw.dz;
  r.ld_dz = bw.ld_dz;
  if ((e = launch_gemm<kModeDZJ>(m.xs, m.wsj, m.xt, m.wtj, r, L)) != cudaSuccess) return e;
  launch_mark(2, L.stream);
  // dxs = dZs Ws (K = V), dWs = dZs^T xs (K = T)
  if ((e = launch_store_gemm<kModeStore>(m.dz, m.ws_mn, T, H, V, dxs, bw.split, g_lse.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(3, L.stream);
  if ((e = launch_store_gemm<kModeStoreT>(m.dz_mn, m.xs_mn, V, H, T, dWs, bw.split, g_lse.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(4, L.stream);
  return cudaSuccess;
}

cudaError_t launch_fljsd_shard_bwd(const FljsdBwdMaps& m, const FusedGeometry& g_jsd, float beta, float inv_tau,
                                   const uint8_t* keep, float grad_scale, const float* lse, const float* kl,
                                   float* dxs, float* dWs, const FusedWs& ws, const FlceBwdWs& bw, float* inv_count,
                                   const FusedLaunch& L) {
  cudaError_t e;
  const int64_t T = g_jsd.T, H = g_jsd.H, V = g_jsd.V;
  launch_mark(0, L.stream);
  // 1 / (kept tokens), then both heads' tiles of this shard again: the student's dZ columns
  if ((e = launch_kept_inv_count(keep, T, inv_count, L.stream)) != cudaSuccess) return e;
  Params r = base_params<kModeDZJ>(g_jsd, L, ws.ctrl);
  r.units = static_cast<int64_t>(r.num_m) * r.num_n;
  r.lse = lse;
  r.beta = beta;
  r.inv_tau = inv_tau;
  r.gscale = grad_scale * inv_tau;
  r.kl = kl;
  r.keep = keep;
  r.inv_count = inv_count;
  r.dz = bw.dz;
  r.ld_dz = bw.ld_dz;
  if ((e = launch_gemm<kModeDZJ>(m.xs, m.wsj, m.xt, m.wtj, r, L)) != cudaSuccess) return e;
  launch_mark(1, L.stream);
  // this shard's share of dxs = dZs Ws_local (K = V_local), its rows of dWs = dZs^T xs (K = T)
  if ((e = launch_store_gemm<kModeStore>(m.dz, m.ws_mn, T, H, V, dxs, bw.split, g_jsd.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(2, L.stream);
  if ((e = launch_store_gemm<kModeStoreT>(m.dz_mn, m.xs_mn, V, H, T, dWs, bw.split, g_jsd.group_store, ws.ctrl, L)) !=
      cudaSuccess)
    return e;
  launch_mark(3, L.stream);
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(Ctrl* ctrl, uint64_t timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lmho
