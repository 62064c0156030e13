// Fused linear + cross-entropy and fused linear + generalized JSD on the
// 5th-generation tensor cores, logits never written to memory.
//
// Operations: page "Fused linear + CPO loss" (summary: activations projected
// through a vocab x hidden LM head, "computed chunked without materializing
// logits"; its cross-entropy core) and page "Fused linear + JSD" (summary:
// student and teacher heads, generalized JSD with beta 0.5, batchmean).
//
// One persistent kernel per pass, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: bf16 tiles x[128 x 64] and W[BN x 64] (128-byte
//               swizzle) into a ring of shared-memory stages (mbarrier
//               complete_tx);
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (M=128, N=BN, K=16, bf16 x bf16 -> fp32) into one of two TMEM
//               accumulators, frees stages with tcgen05.commit;
//   warps 2..5  epilogue: each thread owns one token row (one TMEM lane),
//               reads its accumulator row 32 columns at a time (tcgen05.ld) and
//               folds it into per-row partials while the MMA fills the other
//               accumulator.
// Work unit = (token tile, vocab tile), rastered in groups of `group_m` token
// tiles so a wave of CTAs shares the same W tiles in L2 and each W tile is
// read from HBM about once per group.
//
// Epilogues (per row r of the tile, vocab columns n0 .. n0+BN-1):
//   CE   running (max, sum exp) of the tile and the target logit if t_r falls
//        in the tile  -> partials [num_n][T] x 3
//   LSE  (max, sum exp) only, for the student and teacher heads (first JSD
//        pass)        -> partials [2][num_n][T] x 2
//   JSD  both heads' tiles in TMEM (BN = 128 each); with lp = z_s - lse_s,
//        lq = z_t - lse_t, accumulates
//          beta P (lp - lm) + (1-beta) Q (lq - lm),  lm = ln(beta P + (1-beta) Q)
//        evaluated around the larger of lp, lq so no large terms cancel
//                     -> partial sums [num_n][T]
// Finalisers merge the vocab-tile partials of each row in a fixed order and
// reduce the rows deterministically (see rowstats.cuh).
#include <cmath>
#include <cstdint>

#include "lmho_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace lmho {
namespace {

// CE / LSE / JSD: loss epilogues.  DZ: gradient of the CE with respect to the
// logits, written as bf16 dZ [T, ld_dz] and its transpose dZ^T [V, ld_dzt]
// (inputs of the two backward GEMMs).  STORE: plain fp32 tile store (the
// backward GEMMs dx = dZ W and dW = dZ^T x; rows = T, columns = V in Params).
// JSDK: the divergence pass that also sums KL(P || M) per row (backward only).
// DZJ: both heads recomputed, the student's gradient dZs written like DZ.
enum Mode { kModeCE = 0, kModeLSE = 1, kModeJSD = 2, kModeDZ = 3, kModeStore = 4, kModeJSDK = 5, kModeDZJ = 6 };

template <int MODE>
constexpr bool two_head() { return MODE == kModeJSD || MODE == kModeJSDK || MODE == kModeDZJ; }

constexpr int kTmemCols = 512;   // all of TMEM: accumulators of 256 or 512 fp32 columns
constexpr int kSmemBudget = 192 * 1024;

template <int MODE>
struct ModeCfg {
  static constexpr int BN = two_head<MODE>() ? kBN_JSD : kBN_CE;
  static constexpr int kHeadsPerUnit = two_head<MODE>() ? 2 : 1;
  static constexpr int kAccCols = BN * kHeadsPerUnit;      // TMEM columns of one accumulator
  static constexpr int kNumAcc = kTmemCols / kAccCols;     // 2 = double-buffered, 1 = single
  // Epilogue warps: 4 cover the 128 TMEM lanes; 8 = two per lane quadrant,
  // each taking half of the columns (the two-head epilogue is the heavier one).
  static constexpr int kEpiWarps = two_head<MODE>() ? 4 * kJsdColSplit : 4;
  static constexpr int kColSplit = kEpiWarps / 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;    // producer warp, MMA warp, epilogue
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 512 /*barriers*/;
  static_assert(kNumAcc >= 1 && kNumAcc * kAccCols == kTmemCols, "accumulators tile TMEM");
  static_assert(BN % (32 * kColSplit) == 0, "epilogue column split");
  // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
  // (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
  // N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(kBM >> 4) << 24);
};

struct Params {
  int64_t T, V;
  int32_t num_m, num_n, group_m, k_blocks;
  int64_t units;
  const int64_t* target;  // CE
  float* part0;
  float* part1;
  float* part2;
  const float* lse;  // JSD: [2][T]
  float beta;
  float inv_tau;     // LSE / JSD: logits are multiplied by 1 / temperature
  float gscale;      // DZ: gradient weight of every row (grad_scale / T)
  uint16_t* dz;      // DZ: bf16 [T, ld_dz]
  uint16_t* dzt;     // DZ: bf16 [V, ld_dzt]
  int64_t ld_dz, ld_dzt;
  float* out;        // STORE: fp32 [T, ld_out]
  int64_t ld_out;
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

struct UnitCoord {
  int head;  // LSE: which head; others 0
  int mt, nt;
};

__device__ __forceinline__ UnitCoord decode_unit(const Params& p, int64_t u, int mode) {
  UnitCoord c{0, 0, 0};
  const int64_t per_head = static_cast<int64_t>(p.num_m) * p.num_n;
  if (mode == kModeLSE) {
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

// Generalized-JSD term of one (token, vocab) pair from log-probabilities.
// With hi = max(lp, lq), d = |lp - lq|, e = exp(-d) and weights (w_hi, w_lo)
// the beta weights of the larger and smaller side:
//   lm = hi + ln(w_hi + w_lo e),  hi - lm = -ln(w_hi + w_lo e),  lo - lm = (hi - lm) - d
//   term = w_hi e^hi (hi - lm) + w_lo e^hi e (lo - lm).
__device__ __forceinline__ float jsd_term(float lp, float lq, float beta, float omb) {
  const float hi = fmaxf(lp, lq);
  const float d = fabsf(lp - lq);
  const bool p_is_hi = lp >= lq;
  const float w_hi = p_is_hi ? beta : omb;
  const float w_lo = p_is_hi ? omb : beta;
  const float e = ex2_approx(-d * kLog2e);
  const float a_hi = -kLn2 * lg2_approx(fmaf(w_lo, e, w_hi));
  const float a_lo = a_hi - d;
  const float p_hi = ex2_approx(hi * kLog2e);
  return p_hi * (w_hi * a_hi + w_lo * e * a_lo);
}

// The pieces of one generalized-JSD pair the backward needs: P = e^{lp} and
// lp - lm (same larger-side evaluation as jsd_term).
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
  uint64_t* acc_full = bars + 2 * S;                // [kNumAcc]
  uint64_t* acc_empty = acc_full + C::kNumAcc;      // [kNumAcc]
  uint64_t* drain = acc_empty + C::kNumAcc;         // [1]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::kNumAcc; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::kEpiWarps * 32);
    }
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
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
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
      for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const UnitCoord c = decode_unit(p, u, MODE);
        for (int h = 0; h < C::kHeadsPerUnit && ok; ++h) {
          const int head = (MODE == kModeLSE) ? c.head : h;
          const CUtensorMap* ta = head ? &tm_a1 : &tm_a0;
          const CUtensorMap* tb = head ? &tm_b1 : &tm_b0;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, p.status)) { ok = false; break; }
            uint8_t* sa = tiles + stage * C::kStageBytes;
            uint8_t* sb = sa + C::kABytes;
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
            tma_load_2d(sa, ta, kb * kBK, c.mt * kBM, &full[stage]);
            tma_load_2d(sb, tb, kb * kBK, c.nt * BN, &full[stage]);
            filled |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
      }
      // Never leave with copies in flight: wait for the last fill of each stage.
      for (int s = 0; s < S; ++s)
        if (filled & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, p.timeout_ns, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(tiles);
      for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, p.status)) break;
        tc_fence_after();
        for (int h = 0; h < C::kHeadsPerUnit && ok; ++h) {
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols + h * BN);
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!mbar_wait(&full[stage], phase, p.timeout_ns, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = a0 + stage * C::kStageBytes;
            const uint64_t da = smem_desc_sw128(sa);
            const uint64_t db = smem_desc_sw128(sa + C::kABytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              tc_mma_bf16(d_tmem, da + 2 * k, db + 2 * k, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
            tc_commit(&empty[stage]);
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      tc_commit(drain);
      mbar_wait(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                  // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;            // which column slice (kColSplit slices)
    constexpr int kCols = BN / C::kColSplit;    // columns of each head this warp reads
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    const float beta = p.beta, omb = 1.f - p.beta, it = p.inv_tau;
    for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
      const UnitCoord c = decode_unit(p, u, MODE);
      const int64_t row = static_cast<int64_t>(c.mt) * kBM + row_in_tile;
      const bool row_ok = row < p.T;
      const int64_t n0 = static_cast<int64_t>(c.nt) * BN + half * kCols;
      int64_t tgt = -1;
      float ls = 0.f, lt = 0.f;
      if ((MODE == kModeCE || MODE == kModeDZ) && row_ok) tgt = __ldg(p.target + row);
      if (MODE == kModeDZ && row_ok) ls = __ldg(p.lse + row);
      if (two_head<MODE>() && row_ok) {
        ls = __ldg(p.lse + row);
        lt = __ldg(p.lse + p.T + row);
      }
      float krow = 0.f, gj = 0.f;
      if (MODE == kModeDZJ && row_ok) {
        krow = __ldg(p.kl + row);
        const bool kept = !p.keep || __ldg(p.keep + row);
        gj = kept ? p.gscale * __ldg(p.inv_count) * beta : 0.f;
      }
      // tcgen05.ld is warp-collective: the whole warp proceeds or gives up together
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[acc], acc_phase, p.timeout_ns, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + lane_addr + static_cast<uint32_t>(acc * C::kAccCols + half * kCols);
      MS st = ms_empty();
      float zt = 0.f;
      bool has_t = false;
      float jsd = 0.f, kacc = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < kCols / 32; ++cc) {
        const int64_t col0 = n0 + cc * 32;
        if (MODE == kModeJSDK) {
          float vs[32], vt[32];
          tmem_ld32_sync(tbase + cc * 32, vs);
          tmem_ld32_sync(tbase + BN + cc * 32, vt);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (col0 + j < p.V) {
              const float lp = fmaf(vs[j], it, -ls), lq = fmaf(vt[j], it, -lt);
              float P, lplm;
              jsd_student(lp, lq, beta, omb, &P, &lplm);
              jsd += jsd_term(lp, lq, beta, omb);
              kacc = fmaf(P, lplm, kacc);
            }
          }
        } else if (MODE == kModeDZJ) {
          float vs[32], vt[32];
          tmem_ld32_sync(tbase + cc * 32, vs);
          tmem_ld32_sync(tbase + BN + cc * 32, vt);
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float P, lplm;
              jsd_student(fmaf(vs[j], it, -ls), fmaf(vt[j], it, -lt), beta, omb, &P, &lplm);
              vs[j] = (col0 + j < p.V) ? gj * P * (lplm - krow) : 0.f;
            }
            uint4* dst = reinterpret_cast<uint4*>(p.dz + row * p.ld_dz + col0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(pack_bf16x2(vs[8 * k], vs[8 * k + 1]), pack_bf16x2(vs[8 * k + 2], vs[8 * k + 3]),
                                  pack_bf16x2(vs[8 * k + 4], vs[8 * k + 5]), pack_bf16x2(vs[8 * k + 6], vs[8 * k + 7]));
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < p.V)
                p.dzt[(col0 + j) * p.ld_dzt + row] = static_cast<uint16_t>(pack_bf16x2(vs[j], 0.f));
          }
        } else if (MODE == kModeJSD) {
          float vs[32], vt[32];
          tmem_ld32_sync(tbase + cc * 32, vs);
          tmem_ld32_sync(tbase + BN + cc * 32, vt);
          if (col0 + 32 <= p.V) {
#pragma unroll
            for (int j = 0; j < 32; ++j) jsd += jsd_term(fmaf(vs[j], it, -ls), fmaf(vt[j], it, -lt), beta, omb);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < p.V) jsd += jsd_term(fmaf(vs[j], it, -ls), fmaf(vt[j], it, -lt), beta, omb);
          }
        } else if (MODE == kModeDZ) {
          float v[32];
          tmem_ld32_sync(tbase + cc * 32, v);
          if (row_ok) {
            const bool bad = tgt < 0 || tgt >= p.V;
            const float g = p.gscale, nl = -ls * kLog2e;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t col = col0 + j;
              float d = col < p.V ? g * ex2_approx(fmaf(v[j], kLog2e, nl)) : 0.f;
              if (col == tgt) d -= g;
              v[j] = bad ? __int_as_float(0x7FC00000) : d;
            }
            // dZ row segment: 32 bf16 = 64 contiguous bytes (ld_dz is a multiple of the tile width)
            uint4* dst = reinterpret_cast<uint4*>(p.dz + row * p.ld_dz + col0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                                  pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
            // dZ^T: for each column the 32 lanes (consecutive tokens) write 64 contiguous bytes
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < p.V)
                p.dzt[(col0 + j) * p.ld_dzt + row] = static_cast<uint16_t>(pack_bf16x2(v[j], 0.f));
          }
        } else if (MODE == kModeStore) {
          float v[32];
          tmem_ld32_sync(tbase + cc * 32, v);
          if (row_ok) {
            float* dst = p.out + row * p.ld_out + col0;
            if (col0 + 32 <= p.V) {
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int k = 0; k < 8; ++k) d4[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j < p.V) dst[j] = v[j];
            }
          }
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
          ms_fold<32>(st, v);
        }
      }
      // accumulator fully read: hand it back to the MMA warp
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      if (++acc == C::kNumAcc) { acc = 0; acc_phase ^= 1u; }
      if (row_ok && (MODE == kModeCE || MODE == kModeLSE || MODE == kModeJSD || MODE == kModeJSDK)) {
        // partial slot of this (vocab tile, column slice)
        const int64_t slot = static_cast<int64_t>(c.nt) * C::kColSplit + half;
        if (MODE == kModeJSD || MODE == kModeJSDK) {
          p.part0[slot * p.T + row] = jsd;
          if (MODE == kModeJSDK) p.part1[slot * p.T + row] = kacc;
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
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- finalisers
constexpr int kFinRows = 32;   // rows per block (one per lane)
constexpr int kFinSplit = 8;   // warps per block, each merging a slice of the vocab tiles

// Merge (m, s) partials [num_n][T] of each row, in vocab-tile order, into
// its log-sum-exp.  Warp w handles tiles [w*cnt, (w+1)*cnt); the 8 results
// merge in warp order.
__device__ __forceinline__ float merge_lse_row(const float* pm, const float* ps, int64_t T, int num_n,
                                               int64_t row, MS* s_tmp) {
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
  return tot.m + logf(tot.s);  // meaningful in warp 0
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
  mean_tail(row_out, T, loss, ctrl, gridDim.x, keep, inv_count_out);
}

// out[c, r] = in[r, c] for a bf16 matrix in [rows, cols] (row-major) into
// out [cols, ld_out]; 64 x 64 tiles through shared memory.  Global reads and
// writes move 16 bytes (8 elements) per thread where the tile is whole and
// both sides are 16-byte aligned, element by element otherwise.  Tile rows are
// padded to 72 elements (144 bytes): 16-byte shared stores stay aligned and the
// column reads of 8 consecutive rows fall on distinct banks.
__global__ void __launch_bounds__(256)
    transpose_bf16(const uint16_t* __restrict__ in, int64_t rows, int64_t cols, uint16_t* __restrict__ out,
                   int64_t ld_out) {
  __shared__ __align__(16) uint16_t tile[64][72];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64, c0 = static_cast<int64_t>(blockIdx.x) * 64;
  const bool whole = r0 + 64 <= rows && c0 + 64 <= cols && cols % 8 == 0 && ld_out % 8 == 0 &&
                     (reinterpret_cast<uintptr_t>(in) & 15u) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  if (whole) {
    for (int k = threadIdx.x; k < 512; k += 256) {  // 64 rows x 8 vectors
      const int i = k >> 3, v = k & 7;
      *reinterpret_cast<uint4*>(&tile[i][v * 8]) =
          *reinterpret_cast<const uint4*>(in + (r0 + i) * cols + c0 + v * 8);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < 512; k += 256) {  // 64 output rows (input columns) x 8 vectors
      const int c = k >> 3, v = k & 7;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = static_cast<uint32_t>(tile[v * 8 + 2 * e][c]) | (static_cast<uint32_t>(tile[v * 8 + 2 * e + 1][c]) << 16);
      *reinterpret_cast<uint4*>(out + (c0 + c) * ld_out + r0 + v * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return;
  }
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4 threads
  for (int i = ty; i < 64; i += 4) {
    const int64_t r = r0 + i, c = c0 + tx;
    if (r < rows && c < cols) tile[i][tx] = in[r * cols + c];
  }
  __syncthreads();
  for (int i = ty; i < 64; i += 4) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (c < cols && r < rows) out[c * ld_out + r] = tile[tx][i];
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
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fused_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t grid = p.units < L.num_sms ? p.units : L.num_sms;
  fused_gemm_kernel<MODE><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, L.stream>>>(a0, b0, a1, b1, p);
  return cudaGetLastError();
}

Params base_params(const FusedGeometry& g, const FusedLaunch& L, Ctrl* ctrl) {
  Params p{};
  p.T = g.T;
  p.V = g.V;
  p.num_m = static_cast<int32_t>(g.num_m);
  p.num_n = static_cast<int32_t>(g.num_n);
  p.group_m = g.group_m;
  p.k_blocks = static_cast<int32_t>((g.H + kBK - 1) / kBK);
  p.timeout_ns = L.timeout_ns;
  p.status = &ctrl->status;
  p.inv_tau = 1.f;
  return p;
}

}  // namespace

cudaError_t launch_flce(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const int64_t* target,
                        const FusedGeometry& g, float* loss, const FusedWs& ws, const FusedLaunch& L) {
  Params p = base_params(g, L, ws.ctrl);
  p.units = g.num_m * g.num_n;
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
  Params p = base_params(g_lse, L, ws.ctrl);
  p.units = 2 * g_lse.num_m * g_lse.num_n;
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
  Params q = base_params(g_jsd, L, ws.ctrl);
  q.units = g_jsd.num_m * g_jsd.num_n;
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

cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t rows, int64_t cols, uint16_t* out, int64_t ld_out,
                                  cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
  transpose_bf16<<<grid, 256, 0, st>>>(in, rows, cols, out, ld_out);
  return cudaGetLastError();
}

cudaError_t launch_flce_fwd_bwd(const FlceBwdMaps& m, const uint16_t* x, const uint16_t* W, const int64_t* target,
                                const FusedGeometry& g, float grad_scale, float* loss, float* dx, float* dW,
                                const FusedWs& ws, const FlceBwdWs& bw, const FusedLaunch& L) {
  cudaError_t e;
  launch_mark(0, L.stream);
  // transposed copies so both backward GEMMs read K-major operands
  if ((e = launch_transpose_bf16(W, g.V, g.H, bw.wt, bw.ld_wt, L.stream)) != cudaSuccess) return e;
  if ((e = launch_transpose_bf16(x, g.T, g.H, bw.xt, bw.ld_xt, L.stream)) != cudaSuccess) return e;
  launch_mark(1, L.stream);
  // forward: per-token loss, mean, and each row's log-sum-exp
  Params p = base_params(g, L, ws.ctrl);
  p.units = g.num_m * g.num_n;
  p.target = target;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.part2 = ws.part2;
  if ((e = launch_gemm<kModeCE>(m.x, m.w, m.x, m.w, p, L)) != cudaSuccess) return e;
  const unsigned fblocks = static_cast<unsigned>((g.T + kFinRows - 1) / kFinRows);
  flce_finalize<<<fblocks, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, ws.part2, target, g.T, g.V,
                                                                static_cast<int>(g.num_n), ws.row_out, loss, ws.ctrl,
                                                                bw.lse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  launch_mark(2, L.stream);
  // recompute the logit tiles, write dZ and dZ^T
  Params q = base_params(g, L, ws.ctrl);
  q.units = g.num_m * g.num_n;
  q.target = target;
  q.lse = bw.lse;
  q.gscale = grad_scale / static_cast<float>(g.T);
  q.dz = bw.dz;
  q.dzt = bw.dzt;
  q.ld_dz = bw.ld_dz;
  q.ld_dzt = bw.ld_dzt;
  if ((e = launch_gemm<kModeDZ>(m.x, m.w, m.x, m.w, q, L)) != cudaSuccess) return e;
  launch_mark(3, L.stream);
  // dx [T, H] = dZ [T, V] * W [V, H]   (B operand W^T [H, V], K = V)
  FusedGeometry gx = g;
  gx.T = g.T;
  gx.V = g.H;
  gx.H = g.V;
  gx.num_m = (g.T + kBM - 1) / kBM;
  gx.num_n = (g.H + kBN_CE - 1) / kBN_CE;
  Params a = base_params(gx, L, ws.ctrl);
  a.units = gx.num_m * gx.num_n;
  a.out = dx;
  a.ld_out = g.H;
  if ((e = launch_gemm<kModeStore>(m.dz, m.wt, m.dz, m.wt, a, L)) != cudaSuccess) return e;
  launch_mark(4, L.stream);
  // dW [V, H] = dZ^T [V, T] * x [T, H]   (B operand x^T [H, T], K = T)
  FusedGeometry gw = g;
  gw.T = g.V;
  gw.V = g.H;
  gw.H = g.T;
  gw.num_m = (g.V + kBM - 1) / kBM;
  gw.num_n = (g.H + kBN_CE - 1) / kBN_CE;
  gw.group_m = g.group_m;
  Params b = base_params(gw, L, ws.ctrl);
  b.units = gw.num_m * gw.num_n;
  b.out = dW;
  b.ld_out = g.H;
  if ((e = launch_gemm<kModeStore>(m.dzt, m.xt, m.dzt, m.xt, b, L)) != cudaSuccess) return e;
  launch_mark(5, L.stream);
  return cudaSuccess;
}

cudaError_t launch_fljsd_fwd_bwd(const FljsdBwdMaps& m, const uint16_t* xs, const uint16_t* Ws,
                                 const FusedGeometry& g_lse, const FusedGeometry& g_jsd, float beta, float inv_tau,
                                 const uint8_t* keep, float grad_scale, float* loss, float* dxs, float* dWs,
                                 const FusedWs& ws, const FlceBwdWs& bw, float* kl, float* inv_count,
                                 const FusedLaunch& L) {
  cudaError_t e;
  const int64_t T = g_lse.T, H = g_lse.H, V = g_lse.V;
  launch_mark(0, L.stream);
  if ((e = launch_transpose_bf16(Ws, V, H, bw.wt, bw.ld_wt, L.stream)) != cudaSuccess) return e;
  if ((e = launch_transpose_bf16(xs, T, H, bw.xt, bw.ld_xt, L.stream)) != cudaSuccess) return e;
  launch_mark(1, L.stream);
  // pass 1: log-sum-exp of both heads
  Params p = base_params(g_lse, L, ws.ctrl);
  p.units = 2 * g_lse.num_m * g_lse.num_n;
  p.part0 = ws.part0;
  p.part1 = ws.part1;
  p.inv_tau = inv_tau;
  if ((e = launch_gemm<kModeLSE>(m.xs, m.ws256, m.xt, m.wt256, p, L)) != cudaSuccess) return e;
  dim3 fb(static_cast<unsigned>((T + kFinRows - 1) / kFinRows), 2);
  lse_finalize<<<fb, kFinRows * kFinSplit, 0, L.stream>>>(ws.part0, ws.part1, T, static_cast<int>(g_lse.num_n), ws.lse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // pass 2: divergence and KL(P || M) of every row
  Params q = base_params(g_jsd, L, ws.ctrl);
  q.units = g_jsd.num_m * g_jsd.num_n;
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
  launch_mark(2, L.stream);
  // pass 3: both heads again, the student's dZ and dZ^T
  Params r = base_params(g_jsd, L, ws.ctrl);
  r.units = g_jsd.num_m * g_jsd.num_n;
  r.lse = ws.lse;
  r.beta = beta;
  r.inv_tau = inv_tau;
  r.gscale = grad_scale * inv_tau;
  r.kl = kl;
  r.keep = keep;
  r.inv_count = inv_count;
  r.dz = bw.dz;
  r.dzt = bw.dzt;
  r.ld_dz = bw.ld_dz;
  r.ld_dzt = bw.ld_dzt;
  if ((e = launch_gemm<kModeDZJ>(m.xs, m.wsj, m.xt, m.wtj, r, L)) != cudaSuccess) return e;
  launch_mark(3, L.stream);
  // dxs = dZs Ws, dWs = dZs^T xs
  FusedGeometry gx = g_lse;
  gx.V = H;
  gx.H = V;
  gx.num_m = (T + kBM - 1) / kBM;
  gx.num_n = (H + kBN_CE - 1) / kBN_CE;
  Params a = base_params(gx, L, ws.ctrl);
  a.units = gx.num_m * gx.num_n;
  a.out = dxs;
  a.ld_out = H;
  if ((e = launch_gemm<kModeStore>(m.dz, m.wst, m.dz, m.wst, a, L)) != cudaSuccess) return e;
  launch_mark(4, L.stream);
  FusedGeometry gw = g_lse;
  gw.T = V;
  gw.V = H;
  gw.H = T;
  gw.num_m = (V + kBM - 1) / kBM;
  gw.num_n = (H + kBN_CE - 1) / kBN_CE;
  Params b = base_params(gw, L, ws.ctrl);
  b.units = gw.num_m * gw.num_n;
  b.out = dWs;
  b.ld_out = H;
  if ((e = launch_gemm<kModeStore>(m.dzt, m.xst, m.dzt, m.xst, b, L)) != cudaSuccess) return e;
  launch_mark(5, L.stream);
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(Ctrl* ctrl, uint64_t timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lmho
