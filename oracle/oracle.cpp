// ORACLE -- test infrastructure only.
//
// Plain, slow, obviously-correct fp64 definitions of the losses computed by the
// GPU library.  Only the tests, the package smoke check and the bench's CPU
// baseline leg may load this file's library; the product path never does.  It
// shares no code, header, table or helper with the CUDA sources.
//
// Sources (KernelIndex operation pages; the pages name the losses and give
// their tensor contracts but print no formula, so each definition below is the
// textbook one the names denote):
//   * "Cross-entropy loss", section Semantics: logits float [tokens, vocab],
//     target int64 [tokens], loss float [1]  -> ce_mean_*.
//   * "Vocab-parallel cross-entropy, Megatron layout", summary and Semantics:
//     bf16 logits [seq, batch, vocab], target int64 [seq, batch], per-token fp32
//     loss [seq, batch]; TP = 1 only                    -> ce_sbv_bf16.
//   * "Fused linear + CPO loss", summary ("computed chunked without
//     materializing logits") and Semantics: x [batch, seq, hidden], weight
//     [vocab, hidden], target int64 [batch, seq], loss float [1].  Its
//     cross-entropy (NLL) core -> flce_bf16; the whole CPO objective -> cpo_*
//     (the page names CPO without printing it: the definition below is the
//     published one, Xu et al. 2024, "Contrastive Preference Optimization").
//   * "Fused linear + JSD", summary ("generalized JSD (beta 0.5, batchmean)")
//     and Semantics: student/teacher input [tokens, hidden], student/teacher
//     weight [vocab, hidden], loss float [1]             -> fljsd_bf16.
//
// Definitions (natural log, fp64 throughout, inputs widened exactly):
//   CE row:  loss_i = M_i + ln( sum_v exp(z_iv - M_i) ) - z_{i,t_i},
//            M_i = max_v z_iv, computed as two plain passes over the row.
//            A target outside [0, V) makes that row's loss NaN.
//   mean:    (1/T) sum_i loss_i, summed in row order.
//   fused:   z_iv = sum_k x_ik W_vk (sum in k order), then the CE row.
//   JSD:     P_i = softmax(xs_i Ws^T), Q_i = softmax(xt_i Wt^T),
//            M = beta P + (1-beta) Q,
//            jsd_i = sum_v [ beta P ln(P/M) + (1-beta) Q ln(Q/M) ]
//            (a term whose weight P or Q is 0 contributes 0), and the loss is
//            (1/T) sum_i jsd_i ("batchmean").  P is the student.
//
// Backward of the cross-entropy (gradient of the losses with respect to the
// logits): for row i with upstream weight g_i,
//   dz_iv = g_i * (softmax(z_i)_v - [v == t_i]),  softmax from the two-pass
//   normaliser (exp(z - M) / sum exp(z - M)).
// Flat mean: g_i = scale / T.  Megatron per token: g_i = scale * dloss_i
// (dloss may be null = 1).  A target outside [0, V) makes the row NaN.
//
// CPO: the batch holds 2 Bc sequences of S tokens; sequence b < Bc is the
// chosen answer of pair b and sequence b + Bc its rejected answer.  With the
// per-token CE losses l_{b,s} of the fused linear + CE:
//   lp_b   = -sum_s l_{b,s}                  (sequence log-likelihood)
//   d_k    = lp_k - lp_{k+Bc}
//   pref   = (1/Bc) sum_k -ln sigmoid(beta d_k) = (1/Bc) sum_k softplus(-beta d_k)
//   nll    = (1/(Bc S)) sum_{b < Bc, s} l_{b,s}  (token mean over the chosen half)
//   loss   = alpha nll + pref.
// Its gradient with respect to the per-token losses: alpha/(Bc S) +
// (beta/Bc) sigmoid(-beta d_k) for a chosen token of pair k, and
// -(beta/Bc) sigmoid(-beta d_k) for a rejected one; then the CE backward.

// Vocab-parallel cross-entropy ("Vocab-parallel cross-entropy, Megatron
// layout", summary: the vocabulary split over tensor-parallel ranks, each rank
// holding the logits of its own vocab range, so the local logits are
// [seq, batch, V_local]).  For the shard [v0, v0 + Vl) of row i, two plain
// passes as in the CE row:
//   m_i = max over the shard,  s_i = sum over the shard of exp(z - m_i),
//   zt_i = z_{i, t_i} when v0 <= t_i < v0 + Vl, else -inf.
// Rows of k shards that together cover [0, V) combine, shard by shard in the
// given order, into the row's loss:
//   M = max_j m_j,  loss = M + ln( sum_j s_j exp(m_j - M) ) - max_j zt_j,
// NaN when t_i is outside [0, V).

// Vocab-parallel fused losses (the same vocab split applied to the output
// layer: each rank holds the rows [v0, v0 + Vl) of W, so its logits are
// x W_local^T, [tokens, Vl]):
//   fused CE:  the shard's (m, s, zt) of those logits, combined as above;
//   fused JSD: two combinations.  First each head's log-sum-exp over the
//     shard, l_h = ln sum_{v in shard} exp(z_hv / tau), and the global one
//     lse_h = L + ln( sum_j exp(l_hj - L) ), L = max_j l_hj, in shard order;
//     then, with the global lse, the shard's sum of the JSD terms
//     beta P (lp - ln M) + (1 - beta) Q (lq - ln M), lp = zs/tau - lse_0,
//     lq = zt/tau - lse_1, and the token's JSD is the sum of its shards' sums
//     in shard order (so the split changes only the order of one sum).
//   fused JSD student backward: the shards' shares of each token's
//     KL(P || M) combine by a sum (one more exchange); with the global
//     log-sum-exps and KL, the shard's columns of the student's dz, its share
//     of dxs and its rows of dWs.
//   fused CE backward: with each token's global log-sum-exp (from the
//     gathered partials), the shard's columns of dz = (scale/T)(softmax -
//     onehot); its share dz Wl of dx (the shares sum to dx) and its rows
//     dz^T x of dW.
//
// Variant (JSD with temperature and a token mask): the logits of both heads
// are divided by the temperature tau before the softmax; tokens whose keep
// flag is 0 are left out, and the batchmean divides by the number of kept
// tokens (0 when none is kept).
//
// The thread-count argument of the fused functions only partitions tokens
// across std::threads; each token's arithmetic is the single-threaded code.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNaN = std::numeric_limits<double>::quiet_NaN();

double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Cross-entropy of one row of V logits against target t (two passes).
double ce_row(const double* z, int64_t V, int64_t t) {
  if (t < 0 || t >= V) return kNaN;
  double M = z[0];
  for (int64_t v = 1; v < V; ++v)
    if (z[v] > M || std::isnan(z[v])) M = z[v];
  double sum = 0.0;
  for (int64_t v = 0; v < V; ++v) sum += std::exp(z[v] - M);
  return M + std::log(sum) - z[t];
}

// Log-softmax of one row into lp (lp_v = z_v - logsumexp(z)).
void log_softmax_row(const double* z, int64_t V, double* lp) {
  double M = z[0];
  for (int64_t v = 1; v < V; ++v)
    if (z[v] > M || std::isnan(z[v])) M = z[v];
  double sum = 0.0;
  for (int64_t v = 0; v < V; ++v) sum += std::exp(z[v] - M);
  double lse = M + std::log(sum);
  for (int64_t v = 0; v < V; ++v) lp[v] = z[v] - lse;
}

// Generalized JSD of one token from the two log-probability rows.
double jsd_row(const double* lp, const double* lq, int64_t V, double beta) {
  double acc = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double P = std::exp(lp[v]);
    double Q = std::exp(lq[v]);
    double M = beta * P + (1.0 - beta) * Q;
    double lm = std::log(M);
    double term = 0.0;
    if (P > 0.0) term += beta * P * (lp[v] - lm);
    if (Q > 0.0) term += (1.0 - beta) * Q * (lq[v] - lm);
    acc += term;
  }
  return acc;
}

// z_v = sum_k x_k W_vk for one token (bf16 inputs, exact products in fp64).
void logits_row_bf16(const uint16_t* x, const uint16_t* W, int64_t H, int64_t V, double* z) {
  std::vector<double> xd(H);
  for (int64_t k = 0; k < H; ++k) xd[k] = bf16_to_double(x[k]);
  for (int64_t v = 0; v < V; ++v) {
    const uint16_t* w = W + v * H;
    double acc = 0.0;
    for (int64_t k = 0; k < H; ++k) acc += xd[k] * bf16_to_double(w[k]);
    z[v] = acc;
  }
}

template <class F>
void over_tokens(int64_t T, int threads, F per_token) {
  if (threads <= 1 || T <= 1) {
    for (int64_t i = 0; i < T; ++i) per_token(i);
    return;
  }
  std::vector<std::thread> pool;
  int64_t n = threads < T ? threads : T;
  for (int64_t w = 0; w < n; ++w)
    pool.emplace_back([=] {
      for (int64_t i = w; i < T; i += n) per_token(i);
    });
  for (auto& th : pool) th.join();
}

double mean_of(const double* a, int64_t T) {
  double s = 0.0;
  for (int64_t i = 0; i < T; ++i) s += a[i];
  return s / static_cast<double>(T);
}

}  // namespace

extern "C" {

// Per-row CE over fp64 logits [T, V]; returns the mean, writes per-row losses.
double oracle_ce_f64(const double* z, const int64_t* target, int64_t T, int64_t V,
                     double* loss_rows) {
  for (int64_t i = 0; i < T; ++i) loss_rows[i] = ce_row(z + i * V, V, target[i]);
  return mean_of(loss_rows, T);
}

// Flat layout: fp32 logits [T, V] -> per-row losses and their mean.
double oracle_ce_f32(const float* z32, const int64_t* target, int64_t T, int64_t V,
                     double* loss_rows) {
  std::vector<double> row(V);
  for (int64_t i = 0; i < T; ++i) {
    for (int64_t v = 0; v < V; ++v) row[v] = static_cast<double>(z32[i * V + v]);
    loss_rows[i] = ce_row(row.data(), V, target[i]);
  }
  return mean_of(loss_rows, T);
}

// Megatron layout: bf16 logits [S, B, V] -> per-token losses [S, B] (row s*B+b).
void oracle_ce_sbv_bf16(const uint16_t* z16, const int64_t* target, int64_t S, int64_t B,
                        int64_t V, double* loss_sb) {
  std::vector<double> row(V);
  for (int64_t s = 0; s < S; ++s)
    for (int64_t b = 0; b < B; ++b) {
      int64_t r = s * B + b;
      for (int64_t v = 0; v < V; ++v) row[v] = bf16_to_double(z16[r * V + v]);
      loss_sb[r] = ce_row(row.data(), V, target[r]);
    }
}

// Vocab-parallel CE, one shard: bf16 logits [rows, Vl] holding the global vocab
// columns [v0, v0 + Vl); targets are global indices.  Writes m, s, zt per row.
void oracle_ce_partials_bf16(const uint16_t* z16, const int64_t* target, int64_t rows, int64_t Vl, int64_t v0,
                             double* m_out, double* s_out, double* zt_out) {
  std::vector<double> row(Vl);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t v = 0; v < Vl; ++v) row[v] = bf16_to_double(z16[r * Vl + v]);
    double M = row[0];
    for (int64_t v = 1; v < Vl; ++v)
      if (row[v] > M || std::isnan(row[v])) M = row[v];
    double sum = 0.0;
    for (int64_t v = 0; v < Vl; ++v) sum += std::exp(row[v] - M);
    const int64_t tl = target[r] - v0;
    m_out[r] = M;
    s_out[r] = sum;
    zt_out[r] = (tl >= 0 && tl < Vl) ? row[tl] : -std::numeric_limits<double>::infinity();
  }
}

// The same for the flat layout: fp32 logits [rows, Vl] of the global vocab
// columns [v0, v0 + Vl).
void oracle_ce_partials_f32(const float* z32, const int64_t* target, int64_t rows, int64_t Vl, int64_t v0,
                            double* m_out, double* s_out, double* zt_out) {
  std::vector<double> row(Vl);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t v = 0; v < Vl; ++v) row[v] = static_cast<double>(z32[r * Vl + v]);
    double M = row[0];
    for (int64_t v = 1; v < Vl; ++v)
      if (row[v] > M || std::isnan(row[v])) M = row[v];
    double sum = 0.0;
    for (int64_t v = 0; v < Vl; ++v) sum += std::exp(row[v] - M);
    const int64_t tl = target[r] - v0;
    m_out[r] = M;
    s_out[r] = sum;
    zt_out[r] = (tl >= 0 && tl < Vl) ? row[tl] : -std::numeric_limits<double>::infinity();
  }
}

// Vocab-parallel CE, the combination of k shards' partials (each [k][rows],
// shard-major) into per-row losses; V = the global vocabulary size.
void oracle_ce_merge(const double* m, const double* s, const double* zt, int64_t k, const int64_t* target,
                     int64_t rows, int64_t V, double* loss) {
  for (int64_t r = 0; r < rows; ++r) {
    if (target[r] < 0 || target[r] >= V) {
      loss[r] = kNaN;
      continue;
    }
    double M = m[r];
    double Z = zt[r];
    for (int64_t j = 1; j < k; ++j) {
      if (m[j * rows + r] > M || std::isnan(m[j * rows + r])) M = m[j * rows + r];
      if (zt[j * rows + r] > Z || std::isnan(zt[j * rows + r])) Z = zt[j * rows + r];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < k; ++j) sum += s[j * rows + r] * std::exp(m[j * rows + r] - M);
    loss[r] = M + std::log(sum) - Z;
  }
}

// Fused linear + CE: x [T, H], W [V, H] (bf16) -> per-token losses and their mean.
double oracle_flce_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T,
                        int64_t H, int64_t V, double* loss_rows, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> z(V);
    logits_row_bf16(x + i * H, W, H, V, z.data());
    loss_rows[i] = ce_row(z.data(), V, target[i]);
  });
  return mean_of(loss_rows, T);
}

// Generalized JSD over fp64 student/teacher logits [T, V]; returns batchmean.
double oracle_jsd_f64(const double* zs, const double* zt, int64_t T, int64_t V, double beta,
                      double* jsd_rows) {
  std::vector<double> lp(V), lq(V);
  for (int64_t i = 0; i < T; ++i) {
    log_softmax_row(zs + i * V, V, lp.data());
    log_softmax_row(zt + i * V, V, lq.data());
    jsd_rows[i] = jsd_row(lp.data(), lq.data(), V, beta);
  }
  return mean_of(jsd_rows, T);
}

// Fused linear + generalized JSD (bf16 inputs) -> per-token JSD and batchmean.
double oracle_fljsd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt,
                         const uint16_t* Wt, int64_t T, int64_t H, int64_t V, double beta,
                         double* jsd_rows, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> zs(V), zt(V), lp(V), lq(V);
    logits_row_bf16(xs + i * H, Ws, H, V, zs.data());
    logits_row_bf16(xt + i * H, Wt, H, V, zt.data());
    log_softmax_row(zs.data(), V, lp.data());
    log_softmax_row(zt.data(), V, lq.data());
    jsd_rows[i] = jsd_row(lp.data(), lq.data(), V, beta);
  });
  return mean_of(jsd_rows, T);
}

// Fused linear + generalized JSD with temperature and an optional keep mask
// (keep may be null = every token kept).  jsd_rows gets the per-token JSD
// (0 for tokens left out); returns the mean over kept tokens.
double oracle_fljsd_ex_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt,
                            const uint16_t* Wt, int64_t T, int64_t H, int64_t V, double beta,
                            double tau, const uint8_t* keep, double* jsd_rows, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    if (keep && !keep[i]) {
      jsd_rows[i] = 0.0;
      return;
    }
    std::vector<double> zs(V), zt(V), lp(V), lq(V);
    logits_row_bf16(xs + i * H, Ws, H, V, zs.data());
    logits_row_bf16(xt + i * H, Wt, H, V, zt.data());
    for (int64_t v = 0; v < V; ++v) {
      zs[v] /= tau;
      zt[v] /= tau;
    }
    log_softmax_row(zs.data(), V, lp.data());
    log_softmax_row(zt.data(), V, lq.data());
    jsd_rows[i] = jsd_row(lp.data(), lq.data(), V, beta);
  });
  double sum = 0.0;
  int64_t kept = 0;
  for (int64_t i = 0; i < T; ++i)
    if (!keep || keep[i]) {
      sum += jsd_rows[i];
      ++kept;
    }
  return kept ? sum / static_cast<double>(kept) : 0.0;
}

}  // extern "C"

namespace {
void ce_grad_row(const double* z, int64_t V, int64_t t, double g, double* dz) {
  if (t < 0 || t >= V) {
    for (int64_t v = 0; v < V; ++v) dz[v] = kNaN;
    return;
  }
  double M = z[0];
  for (int64_t v = 1; v < V; ++v)
    if (z[v] > M || std::isnan(z[v])) M = z[v];
  double sum = 0.0;
  for (int64_t v = 0; v < V; ++v) sum += std::exp(z[v] - M);
  for (int64_t v = 0; v < V; ++v) dz[v] = g * (std::exp(z[v] - M) / sum - (v == t ? 1.0 : 0.0));
}
}  // namespace

extern "C" {

// Gradient of the flat mean loss (times scale) w.r.t. fp32 logits [T, V] -> dz [T, V] fp64.
void oracle_ce_grad_f32(const float* z32, const int64_t* target, int64_t T, int64_t V, double scale,
                        double* dz) {
  std::vector<double> row(V);
  const double g = scale / static_cast<double>(T);
  for (int64_t i = 0; i < T; ++i) {
    for (int64_t v = 0; v < V; ++v) row[v] = static_cast<double>(z32[i * V + v]);
    ce_grad_row(row.data(), V, target[i], g, dz + i * V);
  }
}

// Gradient of sum_i dloss_i * loss_i (times scale) w.r.t. fp64 logits [T, V].
void oracle_ce_grad_f64(const double* z, const int64_t* target, int64_t T, int64_t V,
                        const double* dloss, double scale, double* dz) {
  for (int64_t i = 0; i < T; ++i)
    ce_grad_row(z + i * V, V, target[i], scale * (dloss ? dloss[i] : 1.0), dz + i * V);
}

// Megatron layout: bf16 logits [S, B, V], per-token upstream dloss [S, B] (may be
// null) -> dz [S, B, V] fp64.
void oracle_ce_grad_sbv_bf16(const uint16_t* z16, const int64_t* target, int64_t S, int64_t B,
                             int64_t V, const double* dloss, double scale, double* dz) {
  std::vector<double> row(V);
  for (int64_t r = 0; r < S * B; ++r) {
    for (int64_t v = 0; v < V; ++v) row[v] = bf16_to_double(z16[r * V + v]);
    ce_grad_row(row.data(), V, target[r], scale * (dloss ? dloss[r] : 1.0), dz + r * V);
  }
}

// Fused linear + CE on fp64 inputs (for finite-difference pins): x [T, H],
// W [V, H] -> per-token losses, returns the mean.
double oracle_flce_f64(const double* x, const double* W, const int64_t* target, int64_t T, int64_t H,
                       int64_t V, double* loss_rows) {
  std::vector<double> z(V);
  for (int64_t i = 0; i < T; ++i) {
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int64_t k = 0; k < H; ++k) acc += x[i * H + k] * W[v * H + k];
      z[v] = acc;
    }
    loss_rows[i] = ce_row(z.data(), V, target[i]);
  }
  return mean_of(loss_rows, T);
}

// Backward of the fused linear + CE mean (times scale) on fp64 inputs:
//   dZ = (scale / T) (softmax(x W^T) - onehot(t)),  dx = dZ W [T, H],
//   dW = dZ^T x [V, H]  (sums in index order).
void oracle_flce_grad_f64(const double* x, const double* W, const int64_t* target, int64_t T, int64_t H,
                          int64_t V, double scale, double* dx, double* dW) {
  std::vector<double> z(V), dz(static_cast<size_t>(T) * V);
  const double g = scale / static_cast<double>(T);
  for (int64_t i = 0; i < T; ++i) {
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int64_t k = 0; k < H; ++k) acc += x[i * H + k] * W[v * H + k];
      z[v] = acc;
    }
    ce_grad_row(z.data(), V, target[i], g, dz.data() + i * V);
  }
  for (int64_t i = 0; i < T; ++i)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t v = 0; v < V; ++v) acc += dz[i * V + v] * W[v * H + k];
      dx[i * H + k] = acc;
    }
  for (int64_t v = 0; v < V; ++v)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t i = 0; i < T; ++i) acc += dz[i * V + v] * x[i * H + k];
      dW[v * H + k] = acc;
    }
}

// Same from bf16 inputs (widened exactly).
void oracle_flce_grad_bf16(const uint16_t* x16, const uint16_t* W16, const int64_t* target, int64_t T,
                           int64_t H, int64_t V, double scale, double* dx, double* dW) {
  std::vector<double> x(static_cast<size_t>(T) * H), W(static_cast<size_t>(V) * H);
  for (size_t i = 0; i < x.size(); ++i) x[i] = bf16_to_double(x16[i]);
  for (size_t i = 0; i < W.size(); ++i) W[i] = bf16_to_double(W16[i]);
  oracle_flce_grad_f64(x.data(), W.data(), target, T, H, V, scale, dx, dW);
}

// Fused linear + generalized JSD with temperature and keep mask on fp64
// inputs: returns the mean over kept tokens (for finite-difference pins).
double oracle_fljsd_ex_f64(const double* xs, const double* Ws, const double* xt, const double* Wt, int64_t T,
                           int64_t H, int64_t V, double beta, double tau, const uint8_t* keep, double* jsd_rows) {
  std::vector<double> zs(V), zt(V), lp(V), lq(V);
  double sum = 0.0;
  int64_t kept = 0;
  for (int64_t i = 0; i < T; ++i) {
    if (keep && !keep[i]) {
      jsd_rows[i] = 0.0;
      continue;
    }
    for (int64_t v = 0; v < V; ++v) {
      double a = 0.0, b = 0.0;
      for (int64_t k = 0; k < H; ++k) {
        a += xs[i * H + k] * Ws[v * H + k];
        b += xt[i * H + k] * Wt[v * H + k];
      }
      zs[v] = a / tau;
      zt[v] = b / tau;
    }
    log_softmax_row(zs.data(), V, lp.data());
    log_softmax_row(zt.data(), V, lq.data());
    jsd_rows[i] = jsd_row(lp.data(), lq.data(), V, beta);
    sum += jsd_rows[i];
    ++kept;
  }
  return kept ? sum / static_cast<double>(kept) : 0.0;
}

// Student gradients of scale * (the loss above), teacher held fixed.  With
// P = softmax(zs / tau), Q = softmax(zt / tau), M = beta P + (1 - beta) Q:
//   dJSD/dP_v = beta ln(P_v / M_v), so through the softmax
//   dzs_v = (scale / (n_kept tau)) beta P_v (ln P_v - ln M_v - KL(P || M)),
//   dxs = dZs Ws [T, H],  dWs = dZs^T xs [V, H]; left-out tokens give 0 rows.
}  // extern "C"

namespace {
// The student's dZs [T, V] of scale * (fused linear + JSD mean over kept
// tokens) on fp64 inputs (the definition in the comment above); when gbp is
// not null it also receives g beta P [T, V], the factor dZs carries besides
// (ln P - ln M - KL(P || M)).
void fljsd_dz_f64(const double* xs, const double* Ws, const double* xt, const double* Wt, int64_t T, int64_t H,
                  int64_t V, double beta, double tau, const uint8_t* keep, double scale, double* dz,
                  double* gbp = nullptr) {
  int64_t kept = 0;
  for (int64_t i = 0; i < T; ++i) kept += (!keep || keep[i]) ? 1 : 0;
  const double g = kept ? scale / (static_cast<double>(kept) * tau) : 0.0;
  std::vector<double> zs(V), zt(V), lp(V), lq(V), lm(V);
  for (int64_t i = 0; i < T; ++i) {
    if (keep && !keep[i]) {
      for (int64_t v = 0; v < V; ++v) dz[i * V + v] = 0.0;
      if (gbp)
        for (int64_t v = 0; v < V; ++v) gbp[i * V + v] = 0.0;
      continue;
    }
    for (int64_t v = 0; v < V; ++v) {
      double a = 0.0, b = 0.0;
      for (int64_t k = 0; k < H; ++k) {
        a += xs[i * H + k] * Ws[v * H + k];
        b += xt[i * H + k] * Wt[v * H + k];
      }
      zs[v] = a / tau;
      zt[v] = b / tau;
    }
    log_softmax_row(zs.data(), V, lp.data());
    log_softmax_row(zt.data(), V, lq.data());
    double kl = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      lm[v] = std::log(beta * std::exp(lp[v]) + (1.0 - beta) * std::exp(lq[v]));
      kl += std::exp(lp[v]) * (lp[v] - lm[v]);
    }
    for (int64_t v = 0; v < V; ++v) dz[i * V + v] = g * beta * std::exp(lp[v]) * (lp[v] - lm[v] - kl);
    if (gbp)
      for (int64_t v = 0; v < V; ++v) gbp[i * V + v] = g * beta * std::exp(lp[v]);
  }
}
}  // namespace

extern "C" {

void oracle_fljsd_grad_f64(const double* xs, const double* Ws, const double* xt, const double* Wt, int64_t T,
                           int64_t H, int64_t V, double beta, double tau, const uint8_t* keep, double scale,
                           double* dxs, double* dWs) {
  std::vector<double> dz(static_cast<size_t>(T) * V, 0.0);
  fljsd_dz_f64(xs, Ws, xt, Wt, T, H, V, beta, tau, keep, scale, dz.data());
  for (int64_t i = 0; i < T; ++i)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t v = 0; v < V; ++v) acc += dz[i * V + v] * Ws[v * H + k];
      dxs[i * H + k] = acc;
    }
  for (int64_t v = 0; v < V; ++v)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t i = 0; i < T; ++i) acc += dz[i * V + v] * xs[i * H + k];
      dWs[v * H + k] = acc;
    }
}

void oracle_fljsd_grad_bf16(const uint16_t* xs16, const uint16_t* Ws16, const uint16_t* xt16, const uint16_t* Wt16,
                            int64_t T, int64_t H, int64_t V, double beta, double tau, const uint8_t* keep,
                            double scale, double* dxs, double* dWs) {
  std::vector<double> xs(static_cast<size_t>(T) * H), xt(xs.size()), Ws(static_cast<size_t>(V) * H), Wt(Ws.size());
  for (size_t i = 0; i < xs.size(); ++i) {
    xs[i] = bf16_to_double(xs16[i]);
    xt[i] = bf16_to_double(xt16[i]);
  }
  for (size_t i = 0; i < Ws.size(); ++i) {
    Ws[i] = bf16_to_double(Ws16[i]);
    Wt[i] = bf16_to_double(Wt16[i]);
  }
  oracle_fljsd_grad_f64(xs.data(), Ws.data(), xt.data(), Wt.data(), T, H, V, beta, tau, keep, scale, dxs, dWs);
}

// The student's dZs [T, V] (fp64) from bf16 inputs (widened exactly): the
// operand the gradient products multiply, before any rounding; and g beta P.
void oracle_fljsd_dz_bf16(const uint16_t* xs16, const uint16_t* Ws16, const uint16_t* xt16, const uint16_t* Wt16,
                          int64_t T, int64_t H, int64_t V, double beta, double tau, const uint8_t* keep,
                          double scale, double* dz, double* gbp) {
  std::vector<double> xs(static_cast<size_t>(T) * H), xt(xs.size()), Ws(static_cast<size_t>(V) * H), Wt(Ws.size());
  for (size_t i = 0; i < xs.size(); ++i) {
    xs[i] = bf16_to_double(xs16[i]);
    xt[i] = bf16_to_double(xt16[i]);
  }
  for (size_t i = 0; i < Ws.size(); ++i) {
    Ws[i] = bf16_to_double(Ws16[i]);
    Wt[i] = bf16_to_double(Wt16[i]);
  }
  fljsd_dz_f64(xs.data(), Ws.data(), xt.data(), Wt.data(), T, H, V, beta, tau, keep, scale, dz, gbp);
}

// softplus(u) = ln(1 + e^u), and the logistic sigmoid, both without overflow.
static double softplus(double u) { return (u > 0.0 ? u : 0.0) + std::log1p(std::exp(-std::fabs(u))); }
static double sigmoid(double u) {
  if (u >= 0.0) return 1.0 / (1.0 + std::exp(-u));
  const double e = std::exp(u);
  return e / (1.0 + e);
}

// The CPO combination of per-token losses rows [2 Bc * S] (see the header):
// writes lp [2 Bc] (may be null) and sig [Bc] = sigmoid(-beta d_k) (may be
// null), returns the loss.  Sums run in index order.
static double cpo_combine(const double* rows, int64_t B, int64_t S, double beta, double alpha, double* lp, double* sig) {
  const int64_t Bc = B / 2;
  std::vector<double> seq(B);
  for (int64_t b = 0; b < B; ++b) {
    double acc = 0.0;
    for (int64_t s = 0; s < S; ++s) acc += rows[b * S + s];
    seq[b] = -acc;
    if (lp) lp[b] = seq[b];
  }
  double pref = 0.0, nll = 0.0;
  for (int64_t k = 0; k < Bc; ++k) {
    const double d = seq[k] - seq[k + Bc];
    pref += softplus(-beta * d);
    if (sig) sig[k] = sigmoid(-beta * d);
    nll -= seq[k];
  }
  return alpha * nll / (static_cast<double>(Bc) * S) + pref / static_cast<double>(Bc);
}

// d loss / d l_i of a token of sequence b (see the header): sig = sigmoid(-beta d_k) of its pair.
static double cpo_row_weight(int64_t b, int64_t S, int64_t Bc, double beta, double alpha, const double* sig) {
  return b < Bc ? alpha / (static_cast<double>(Bc) * S) + beta / Bc * sig[b] : -beta / Bc * sig[b - Bc];
}

// The CPO combination alone, from given per-token losses rows [B*S]: writes
// lp [B] and the per-token weights d loss / d l_i into row_w [B*S] (may be
// null); returns the loss.  Lets tests check large cases from sampled rows.
double oracle_cpo_combine(const double* rows, int64_t B, int64_t S, double beta, double alpha, double* lp,
                          double* row_w) {
  std::vector<double> sig(B / 2);
  const double m = cpo_combine(rows, B, S, beta, alpha, lp, sig.data());
  if (row_w)
    for (int64_t i = 0; i < B * S; ++i) row_w[i] = cpo_row_weight(i / S, S, B / 2, beta, alpha, sig.data());
  return m;
}

// CPO on the fused linear + CE, fp64 inputs x [B*S, H], W [V, H]: per-token
// CE losses into loss_rows [B*S], sequence log-likelihoods into lp [B] (may
// be null); returns the loss.
double oracle_cpo_f64(const double* x, const double* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                      int64_t V, double beta, double alpha, double* loss_rows, double* lp) {
  oracle_flce_f64(x, W, target, B * S, H, V, loss_rows);
  return cpo_combine(loss_rows, B, S, beta, alpha, lp, nullptr);
}

// Same from bf16 inputs; the per-token losses come from oracle_flce_bf16
// (threads only partition tokens).
double oracle_cpo_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B, int64_t S,
                       int64_t H, int64_t V, double beta, double alpha, double* loss_rows, double* lp,
                       int threads) {
  oracle_flce_bf16(x, W, target, B * S, H, V, loss_rows, threads);
  return cpo_combine(loss_rows, B, S, beta, alpha, lp, nullptr);
}

// Gradient of scale * (CPO loss) on fp64 inputs:
//   dz_i = scale w_i (softmax(z_i) - onehot(t_i)),  w_i as in the header,
//   dx = dZ W [B*S, H],  dW = dZ^T x [V, H]  (sums in index order).
void oracle_cpo_grad_f64(const double* x, const double* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                         int64_t V, double beta, double alpha, double scale, double* dx, double* dW) {
  const int64_t T = B * S, Bc = B / 2;
  std::vector<double> rows(T), sig(Bc), z(V), dz(static_cast<size_t>(T) * V);
  oracle_flce_f64(x, W, target, T, H, V, rows.data());
  cpo_combine(rows.data(), B, S, beta, alpha, nullptr, sig.data());
  for (int64_t i = 0; i < T; ++i) {
    const double w = cpo_row_weight(i / S, S, Bc, beta, alpha, sig.data());
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int64_t kk = 0; kk < H; ++kk) acc += x[i * H + kk] * W[v * H + kk];
      z[v] = acc;
    }
    ce_grad_row(z.data(), V, target[i], scale * w, dz.data() + i * V);
  }
  for (int64_t i = 0; i < T; ++i)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t v = 0; v < V; ++v) acc += dz[i * V + v] * W[v * H + k];
      dx[i * H + k] = acc;
    }
  for (int64_t v = 0; v < V; ++v)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t i = 0; i < T; ++i) acc += dz[i * V + v] * x[i * H + k];
      dW[v * H + k] = acc;
    }
}

void oracle_cpo_grad_bf16(const uint16_t* x16, const uint16_t* W16, const int64_t* target, int64_t B, int64_t S,
                          int64_t H, int64_t V, double beta, double alpha, double scale, double* dx, double* dW) {
  std::vector<double> x(static_cast<size_t>(B * S) * H), W(static_cast<size_t>(V) * H);
  for (size_t i = 0; i < x.size(); ++i) x[i] = bf16_to_double(x16[i]);
  for (size_t i = 0; i < W.size(); ++i) W[i] = bf16_to_double(W16[i]);
  oracle_cpo_grad_f64(x.data(), W.data(), target, B, S, H, V, beta, alpha, scale, dx, dW);
}

// Logits of the fused paths for a set of tokens (used by tests to pin the
// fused functions against ce on explicit logits): z [T, V].
void oracle_logits_bf16(const uint16_t* x, const uint16_t* W, int64_t T, int64_t H, int64_t V,
                        double* z) {
  for (int64_t i = 0; i < T; ++i) logits_row_bf16(x + i * H, W, H, V, z + i * V);
}

// Vocab-parallel fused linear + CE, one shard: x [T, H], Wl [Vl, H] (bf16) =
// the global vocab rows [v0, v0 + Vl); targets are global.  The shard's max m,
// sum of exp(z - m) s and target logit zt (-inf when the target is not in the
// shard) of each token's logits x_i Wl^T, two plain passes as in ce_row.
void oracle_flce_partials_bf16(const uint16_t* x, const uint16_t* Wl, const int64_t* target, int64_t T, int64_t H,
                               int64_t Vl, int64_t v0, double* m_out, double* s_out, double* zt_out, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> z(Vl);
    logits_row_bf16(x + i * H, Wl, H, Vl, z.data());
    double M = z[0];
    for (int64_t v = 1; v < Vl; ++v)
      if (z[v] > M || std::isnan(z[v])) M = z[v];
    double sum = 0.0;
    for (int64_t v = 0; v < Vl; ++v) sum += std::exp(z[v] - M);
    const int64_t tl = target[i] - v0;
    m_out[i] = M;
    s_out[i] = sum;
    zt_out[i] = (tl >= 0 && tl < Vl) ? z[tl] : -std::numeric_limits<double>::infinity();
  });
}

// Vocab-parallel fused linear + JSD, first combination, one shard: each head's
// log-sum-exp over the shard's columns of the logits divided by tau; lse [2][T]
// (head 0 = student xs Wsl^T, head 1 = teacher xt Wtl^T).
void oracle_fljsd_lse_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                 int64_t T, int64_t H, int64_t Vl, double tau, double* lse, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> z(Vl);
    for (int h = 0; h < 2; ++h) {
      logits_row_bf16((h ? xt : xs) + i * H, h ? Wtl : Wsl, H, Vl, z.data());
      for (int64_t v = 0; v < Vl; ++v) z[v] /= tau;
      double M = z[0];
      for (int64_t v = 1; v < Vl; ++v)
        if (z[v] > M || std::isnan(z[v])) M = z[v];
      double sum = 0.0;
      for (int64_t v = 0; v < Vl; ++v) sum += std::exp(z[v] - M);
      lse[h * T + i] = M + std::log(sum);
    }
  });
}

// The global log-sum-exps [2][T] from k shards' [k][2][T] (shard-major), in
// shard order: L = max_j l_j, lse = L + ln sum_j exp(l_j - L).
void oracle_lse_merge(const double* parts, int64_t k, int64_t T, double* lse) {
  for (int64_t h = 0; h < 2; ++h)
    for (int64_t i = 0; i < T; ++i) {
      double L = parts[h * T + i];
      for (int64_t j = 1; j < k; ++j) {
        const double l = parts[(j * 2 + h) * T + i];
        if (l > L || std::isnan(l)) L = l;
      }
      double sum = 0.0;
      for (int64_t j = 0; j < k; ++j) sum += std::exp(parts[(j * 2 + h) * T + i] - L);
      lse[h * T + i] = L + std::log(sum);
    }
}

// Vocab-parallel fused linear + JSD, second combination, one shard: with the
// global log-sum-exps lse [2][T], each token's sum over the shard's columns of
// the generalized JSD terms (jsd_row on the shard's log-probabilities).
void oracle_fljsd_terms_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                   int64_t T, int64_t H, int64_t Vl, double beta, double tau, const double* lse,
                                   double* terms, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> lp(Vl), lq(Vl);
    logits_row_bf16(xs + i * H, Wsl, H, Vl, lp.data());
    logits_row_bf16(xt + i * H, Wtl, H, Vl, lq.data());
    for (int64_t v = 0; v < Vl; ++v) {
      lp[v] = lp[v] / tau - lse[i];
      lq[v] = lq[v] / tau - lse[T + i];
    }
    terms[i] = jsd_row(lp.data(), lq.data(), Vl, beta);
  });
}

// Each row's global log-sum-exp from k shards' CE partials (each [k][rows],
// shard-major): M = max_j m_j, lse = M + ln sum_j s_j exp(m_j - M).
void oracle_ce_partials_lse(const double* m, const double* s, int64_t k, int64_t rows, double* lse) {
  for (int64_t r = 0; r < rows; ++r) {
    double M = m[r];
    for (int64_t j = 1; j < k; ++j)
      if (m[j * rows + r] > M || std::isnan(m[j * rows + r])) M = m[j * rows + r];
    double sum = 0.0;
    for (int64_t j = 0; j < k; ++j) sum += s[j * rows + r] * std::exp(m[j * rows + r] - M);
    lse[r] = M + std::log(sum);
  }
}

// Backward of one shard of the vocab-parallel fused linear + CE (W rows
// [v0, v0 + Vl) in Wl), gradient of scale * mean loss over the T tokens:
//   dz_iv = (scale / T) (exp(z_iv - lse_i) - [v0 + v == t_i]) for the shard's
//   columns v, lse_i the token's global log-sum-exp; a target outside [0, V)
//   makes the row NaN;
//   dx_partial = dz Wl [T, H] (the shards' shares sum to dx), dWl = dz^T x [Vl, H].
void oracle_flce_grad_shard_bf16(const uint16_t* x16, const uint16_t* Wl16, const int64_t* target, int64_t T,
                                 int64_t H, int64_t Vl, int64_t v0, int64_t V, const double* lse, double scale,
                                 double* dx, double* dWl) {
  std::vector<double> x(static_cast<size_t>(T) * H), W(static_cast<size_t>(Vl) * H), dz(static_cast<size_t>(T) * Vl);
  for (size_t i = 0; i < x.size(); ++i) x[i] = bf16_to_double(x16[i]);
  for (size_t i = 0; i < W.size(); ++i) W[i] = bf16_to_double(Wl16[i]);
  const double g = scale / static_cast<double>(T);
  for (int64_t i = 0; i < T; ++i) {
    const bool bad = target[i] < 0 || target[i] >= V;
    for (int64_t v = 0; v < Vl; ++v) {
      double z = 0.0;
      for (int64_t k = 0; k < H; ++k) z += x[i * H + k] * W[v * H + k];
      dz[i * Vl + v] = bad ? kNaN : g * (std::exp(z - lse[i]) - (v0 + v == target[i] ? 1.0 : 0.0));
    }
  }
  for (int64_t i = 0; i < T; ++i)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t v = 0; v < Vl; ++v) acc += dz[i * Vl + v] * W[v * H + k];
      dx[i * H + k] = acc;
    }
  for (int64_t v = 0; v < Vl; ++v)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t i = 0; i < T; ++i) acc += dz[i * Vl + v] * x[i * H + k];
      dWl[v * H + k] = acc;
    }
}

// Vocab-parallel fused linear + JSD, the student backward of one shard
// (student rows Wsl, teacher rows Wtl [Vl, H]), with the global log-sum-exps
// lse [2][T] of the logits / tau:
//   lp = zs/tau - lse_0, lq = zt/tau - lse_1, P = e^lp, lm = ln(beta P + (1-beta) e^lq);
//   kl_i = sum over the shard's columns of P (lp - lm): the shard's share of
//   KL(P || M) (the shares sum to it).
void oracle_fljsd_kl_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                int64_t T, int64_t H, int64_t Vl, double beta, double tau, const double* lse,
                                double* kl, int threads) {
  over_tokens(T, threads, [&](int64_t i) {
    std::vector<double> zs(Vl), zt(Vl);
    logits_row_bf16(xs + i * H, Wsl, H, Vl, zs.data());
    logits_row_bf16(xt + i * H, Wtl, H, Vl, zt.data());
    double acc = 0.0;
    for (int64_t v = 0; v < Vl; ++v) {
      const double lp = zs[v] / tau - lse[i], lq = zt[v] / tau - lse[T + i];
      const double lm = std::log(beta * std::exp(lp) + (1.0 - beta) * std::exp(lq));
      acc += std::exp(lp) * (lp - lm);
    }
    kl[i] = acc;
  });
}

// ... and with each token's global KL(P || M) kl [T]: the shard's columns of
//   dz_iv = g beta P (lp - lm - kl_i),  g = scale / (n_kept tau),
// rows of tokens whose keep flag is 0 are 0 (keep may be null = all kept, a
// batch with no kept token has g = 0); dxs = dz Wsl [T, H] (the shards' shares
// sum to the student's dx), dWsl = dz^T xs [Vl, H] (its rows of dW).
void oracle_fljsd_grad_shard_bf16(const uint16_t* xs16, const uint16_t* Wsl16, const uint16_t* xt16,
                                  const uint16_t* Wtl16, int64_t T, int64_t H, int64_t Vl, double beta, double tau,
                                  const uint8_t* keep, const double* lse, const double* kl, double scale, double* dxs,
                                  double* dWsl) {
  std::vector<double> xs(static_cast<size_t>(T) * H), Ws(static_cast<size_t>(Vl) * H),
      dz(static_cast<size_t>(T) * Vl, 0.0);
  for (size_t i = 0; i < xs.size(); ++i) xs[i] = bf16_to_double(xs16[i]);
  for (size_t i = 0; i < Ws.size(); ++i) Ws[i] = bf16_to_double(Wsl16[i]);
  int64_t kept = 0;
  for (int64_t i = 0; i < T; ++i) kept += (!keep || keep[i]) ? 1 : 0;
  const double g = kept ? scale / (static_cast<double>(kept) * tau) : 0.0;
  std::vector<double> zs(Vl), zt(Vl);
  for (int64_t i = 0; i < T; ++i) {
    if (keep && !keep[i]) continue;
    logits_row_bf16(xs16 + i * H, Wsl16, H, Vl, zs.data());
    logits_row_bf16(xt16 + i * H, Wtl16, H, Vl, zt.data());
    for (int64_t v = 0; v < Vl; ++v) {
      const double lp = zs[v] / tau - lse[i], lq = zt[v] / tau - lse[T + i];
      const double lm = std::log(beta * std::exp(lp) + (1.0 - beta) * std::exp(lq));
      dz[i * Vl + v] = g * beta * std::exp(lp) * (lp - lm - kl[i]);
    }
  }
  for (int64_t i = 0; i < T; ++i)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t v = 0; v < Vl; ++v) acc += dz[i * Vl + v] * Ws[v * H + k];
      dxs[i * H + k] = acc;
    }
  for (int64_t v = 0; v < Vl; ++v)
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t i = 0; i < T; ++i) acc += dz[i * Vl + v] * xs[i * H + k];
      dWsl[v * H + k] = acc;
    }
}

// The per-token JSD from k shards' term sums [k][T] (summed in shard order; 0
// for tokens whose keep flag is 0, keep may be null) and their batchmean over
// the kept tokens (0 when none is kept).
double oracle_jsd_merge(const double* terms, int64_t k, int64_t T, const uint8_t* keep, double* rows) {
  double total = 0.0;
  int64_t kept = 0;
  for (int64_t i = 0; i < T; ++i) {
    if (keep && !keep[i]) {
      rows[i] = 0.0;
      continue;
    }
    double acc = 0.0;
    for (int64_t j = 0; j < k; ++j) acc += terms[j * T + i];
    rows[i] = acc;
    total += acc;
    ++kept;
  }
  return kept ? total / static_cast<double>(kept) : 0.0;
}

}  // extern "C"
