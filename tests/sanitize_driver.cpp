// Test driver for the host-side C++ (the fp64 oracle and the input generator)
// built with AddressSanitizer and UndefinedBehaviorSanitizer: it calls every
// exported routine on small ragged shapes, with several threads where the
// routine takes a thread count, plus the edge cases the tests use (an
// out-of-range target, a keep mask, V = 1).  It checks nothing numerically --
// the pytest pins do that -- it only gives the sanitizers every code path.
// Exit status 0 = clean (the sanitizers abort with a report otherwise).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>

extern "C" {
void gen_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void gen_normal_f64(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n, double sigma, double* out,
                    int threads);
void gen_normal_f32(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n, double sigma, float* out,
                    int threads);
void gen_normal_bf16(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n, double sigma, uint16_t* out,
                     int threads);
void gen_targets(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n, int64_t V, int64_t* out,
                 int threads);

double oracle_ce_f64(const double* z, const int64_t* target, int64_t T, int64_t V, double* loss_rows);
double oracle_ce_f32(const float* z32, const int64_t* target, int64_t T, int64_t V, double* loss_rows);
void oracle_ce_sbv_bf16(const uint16_t* z16, const int64_t* target, int64_t S, int64_t B, int64_t V,
                        double* loss_sb);
double oracle_flce_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T, int64_t H,
                        int64_t V, double* loss_rows, int threads);
double oracle_jsd_f64(const double* zs, const double* zt, int64_t T, int64_t V, double beta, double* jsd_rows);
double oracle_fljsd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T,
                         int64_t H, int64_t V, double beta, double* jsd_rows, int threads);
double oracle_fljsd_ex_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt,
                            int64_t T, int64_t H, int64_t V, double beta, double tau, const uint8_t* keep,
                            double* jsd_rows, int threads);
void oracle_ce_grad_f32(const float* z32, const int64_t* target, int64_t T, int64_t V, double scale, double* dz);
void oracle_ce_grad_f64(const double* z, const int64_t* target, int64_t T, int64_t V, const double* dloss,
                        double scale, double* dz);
void oracle_ce_grad_sbv_bf16(const uint16_t* z16, const int64_t* target, int64_t S, int64_t B, int64_t V,
                             const double* dloss, double scale, double* dz);
double oracle_flce_f64(const double* x, const double* W, const int64_t* target, int64_t T, int64_t H, int64_t V,
                       double* loss_rows);
void oracle_flce_grad_f64(const double* x, const double* W, const int64_t* target, int64_t T, int64_t H, int64_t V,
                          double scale, double* dx, double* dW);
void oracle_flce_grad_bf16(const uint16_t* x16, const uint16_t* W16, const int64_t* target, int64_t T, int64_t H,
                           int64_t V, double scale, double* dx, double* dW);
double oracle_fljsd_ex_f64(const double* xs, const double* Ws, const double* xt, const double* Wt, int64_t T,
                           int64_t H, int64_t V, double beta, double tau, const uint8_t* keep, double* jsd_rows);
void oracle_fljsd_grad_f64(const double* xs, const double* Ws, const double* xt, const double* Wt, int64_t T,
                           int64_t H, int64_t V, double beta, double tau, const uint8_t* keep, double scale,
                           double* dxs, double* dWs);
void oracle_fljsd_grad_bf16(const uint16_t* xs16, const uint16_t* Ws16, const uint16_t* xt16, const uint16_t* Wt16,
                            int64_t T, int64_t H, int64_t V, double beta, double tau, const uint8_t* keep,
                            double scale, double* dxs, double* dWs);
double oracle_cpo_combine(const double* rows, int64_t B, int64_t S, double beta, double alpha, double* lp,
                          double* row_w);
double oracle_cpo_f64(const double* x, const double* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                      int64_t V, double beta, double alpha, double* loss_rows, double* lp);
double oracle_cpo_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                       int64_t V, double beta, double alpha, double* loss_rows, double* lp, int threads);
void oracle_cpo_grad_f64(const double* x, const double* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                         int64_t V, double beta, double alpha, double scale, double* dx, double* dW);
void oracle_cpo_grad_bf16(const uint16_t* x16, const uint16_t* W16, const int64_t* target, int64_t B, int64_t S,
                          int64_t H, int64_t V, double beta, double alpha, double scale, double* dx, double* dW);
void oracle_logits_bf16(const uint16_t* x, const uint16_t* W, int64_t T, int64_t H, int64_t V, double* z);
void oracle_ce_partials_bf16(const uint16_t* z16, const int64_t* target, int64_t rows, int64_t Vl, int64_t v0,
                             double* m_out, double* s_out, double* zt_out);
void oracle_ce_partials_f32(const float* z32, const int64_t* target, int64_t rows, int64_t Vl, int64_t v0,
                            double* m_out, double* s_out, double* zt_out);
void oracle_ce_merge(const double* m, const double* s, const double* zt, int64_t k, const int64_t* target,
                     int64_t rows, int64_t V, double* loss);
void oracle_fljsd_dz_bf16(const uint16_t* xs16, const uint16_t* Ws16, const uint16_t* xt16, const uint16_t* Wt16,
                          int64_t T, int64_t H, int64_t V, double beta, double tau, const uint8_t* keep,
                          double scale, double* dz, double* gbp);
void oracle_flce_partials_bf16(const uint16_t* x, const uint16_t* Wl, const int64_t* target, int64_t T, int64_t H,
                               int64_t Vl, int64_t v0, double* m_out, double* s_out, double* zt_out, int threads);
void oracle_fljsd_lse_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                 int64_t T, int64_t H, int64_t Vl, double tau, double* lse, int threads);
void oracle_lse_merge(const double* parts, int64_t k, int64_t T, double* lse);
void oracle_fljsd_terms_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                   int64_t T, int64_t H, int64_t Vl, double beta, double tau, const double* lse,
                                   double* terms, int threads);
double oracle_jsd_merge(const double* terms, int64_t k, int64_t T, const uint8_t* keep, double* rows);
void oracle_ce_partials_lse(const double* m, const double* s, int64_t k, int64_t rows, double* lse);
void oracle_fljsd_kl_shard_bf16(const uint16_t* xs, const uint16_t* Wsl, const uint16_t* xt, const uint16_t* Wtl,
                                int64_t T, int64_t H, int64_t Vl, double beta, double tau, const double* lse,
                                double* kl, int threads);
void oracle_fljsd_grad_shard_bf16(const uint16_t* xs16, const uint16_t* Wsl16, const uint16_t* xt16,
                                  const uint16_t* Wtl16, int64_t T, int64_t H, int64_t Vl, double beta, double tau,
                                  const uint8_t* keep, const double* lse, const double* kl, double scale, double* dxs,
                                  double* dWsl);
void oracle_flce_grad_shard_bf16(const uint16_t* x16, const uint16_t* Wl16, const int64_t* target, int64_t T,
                                 int64_t H, int64_t Vl, int64_t v0, int64_t V, const double* lse, double scale,
                                 double* dx, double* dWl);
}

namespace {

// One shape through every routine.  B = 2 sequences of S = T / 2 tokens for CPO.
void run_shape(int64_t T, int64_t H, int64_t V, int threads) {
  const uint64_t seed = 1000 + static_cast<uint64_t>(T * 7 + H * 3 + V);
  std::vector<double> zd(T * V), zd2(T * V), xd(T * H), Wd(V * H), xd2(T * H), Wd2(V * H);
  std::vector<float> zf(T * V);
  std::vector<uint16_t> zb(T * V), xb(T * H), Wb(V * H), xb2(T * H), Wb2(V * H);
  std::vector<int64_t> t(T);
  gen_normal_f64(seed, 0, 0, zd.size(), 2.0, zd.data(), threads);
  gen_normal_f64(seed, 3, 0, zd2.size(), 2.0, zd2.data(), threads);
  gen_normal_f32(seed, 0, 5, zf.size(), 1.0, zf.data(), threads);
  gen_normal_bf16(seed, 0, 0, zb.size(), 2.0, zb.data(), threads);
  gen_normal_f64(seed, 0, 0, xd.size(), 1.0, xd.data(), threads);
  gen_normal_f64(seed, 2, 0, Wd.size(), 0.3, Wd.data(), threads);
  gen_normal_f64(seed, 3, 0, xd2.size(), 1.0, xd2.data(), threads);
  gen_normal_f64(seed, 4, 0, Wd2.size(), 0.3, Wd2.data(), threads);
  gen_normal_bf16(seed, 0, 0, xb.size(), 1.0, xb.data(), threads);
  gen_normal_bf16(seed, 2, 0, Wb.size(), 0.3, Wb.data(), threads);
  gen_normal_bf16(seed, 3, 0, xb2.size(), 1.0, xb2.data(), threads);
  gen_normal_bf16(seed, 4, 0, Wb2.size(), 0.3, Wb2.data(), threads);
  gen_targets(seed, 1, 0, t.size(), V, t.data(), threads);
  if (T > 1) t[1] = V;  // an out-of-range target: NaN for that token, no out-of-bounds access

  std::vector<double> rows(T), rows2(T), dz(T * V), dx(T * H), dW(V * H), lp(2), w(T), zl(T * V), dloss(T, 0.5);
  std::vector<uint8_t> keep(T);
  for (int64_t i = 0; i < T; ++i) keep[i] = static_cast<uint8_t>(i % 3 != 0);

  oracle_ce_f64(zd.data(), t.data(), T, V, rows.data());
  oracle_ce_f32(zf.data(), t.data(), T, V, rows.data());
  oracle_ce_sbv_bf16(zb.data(), t.data(), T, 1, V, rows.data());
  oracle_flce_bf16(xb.data(), Wb.data(), t.data(), T, H, V, rows.data(), threads);
  oracle_jsd_f64(zd.data(), zd2.data(), T, V, 0.5, rows.data());
  oracle_fljsd_bf16(xb.data(), Wb.data(), xb2.data(), Wb2.data(), T, H, V, 0.3, rows.data(), threads);
  oracle_fljsd_ex_bf16(xb.data(), Wb.data(), xb2.data(), Wb2.data(), T, H, V, 0.7, 2.0, keep.data(), rows.data(),
                       threads);
  oracle_fljsd_ex_bf16(xb.data(), Wb.data(), xb2.data(), Wb2.data(), T, H, V, 0.5, 1.0, nullptr, rows.data(),
                       threads);
  oracle_ce_grad_f32(zf.data(), t.data(), T, V, 1.5, dz.data());
  oracle_ce_grad_f64(zd.data(), t.data(), T, V, dloss.data(), 1.0, dz.data());
  oracle_ce_grad_f64(zd.data(), t.data(), T, V, nullptr, 1.0, dz.data());
  oracle_ce_grad_sbv_bf16(zb.data(), t.data(), T, 1, V, dloss.data(), 2.0, dz.data());
  oracle_flce_f64(xd.data(), Wd.data(), t.data(), T, H, V, rows.data());
  oracle_flce_grad_f64(xd.data(), Wd.data(), t.data(), T, H, V, 1.0, dx.data(), dW.data());
  oracle_flce_grad_bf16(xb.data(), Wb.data(), t.data(), T, H, V, 3.0, dx.data(), dW.data());
  oracle_fljsd_ex_f64(xd.data(), Wd.data(), xd2.data(), Wd2.data(), T, H, V, 0.5, 1.0, keep.data(), rows.data());
  oracle_fljsd_grad_f64(xd.data(), Wd.data(), xd2.data(), Wd2.data(), T, H, V, 0.3, 0.8, keep.data(), 1.0, dx.data(),
                        dW.data());
  oracle_fljsd_grad_bf16(xb.data(), Wb.data(), xb2.data(), Wb2.data(), T, H, V, 0.5, 1.0, nullptr, 2.0, dx.data(),
                         dW.data());
  oracle_logits_bf16(xb.data(), Wb.data(), T, H, V, zl.data());
  oracle_fljsd_dz_bf16(xb.data(), Wb.data(), xb2.data(), Wb2.data(), T, H, V, 0.3, 2.0, keep.data(), 1.0, dz.data(),
                       zl.data());
  // vocab-parallel: split V into up to three shards (each its own [T, w] buffer), merge
  {
    const int64_t k = V >= 3 ? 3 : V;
    std::vector<double> m(k * T), sm(k * T), zt(k * T);
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      std::vector<uint16_t> local(T * w1);
      for (int64_t i = 0; i < T; ++i)
        for (int64_t v = 0; v < w1; ++v) local[i * w1 + v] = zb[i * V + v0 + v];
      oracle_ce_partials_bf16(local.data(), t.data(), T, w1, v0, m.data() + j * T, sm.data() + j * T,
                              zt.data() + j * T);
    }
    oracle_ce_merge(m.data(), sm.data(), zt.data(), k, t.data(), T, V, rows.data());
    for (int64_t j = 0; j < k; ++j) {   // the flat fp32 layout
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      std::vector<float> local(T * w1);
      for (int64_t i = 0; i < T; ++i)
        for (int64_t v = 0; v < w1; ++v) local[i * w1 + v] = zf[i * V + v0 + v];
      oracle_ce_partials_f32(local.data(), t.data(), T, w1, v0, m.data() + j * T, sm.data() + j * T,
                             zt.data() + j * T);
    }
    oracle_ce_merge(m.data(), sm.data(), zt.data(), k, t.data(), T, V, rows.data());
    // the fused forms: shards of W's rows, each its own [w, H] slice of the same buffer
    std::vector<double> lparts(k * 2 * T), lse(2 * T), terms(k * T);
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      oracle_flce_partials_bf16(xb.data(), Wb.data() + v0 * H, t.data(), T, H, w1, v0, m.data() + j * T,
                                sm.data() + j * T, zt.data() + j * T, threads);
      oracle_fljsd_lse_shard_bf16(xb.data(), Wb.data() + v0 * H, xb2.data(), Wb2.data() + v0 * H, T, H, w1, 1.5,
                                  lparts.data() + j * 2 * T, threads);
    }
    oracle_ce_merge(m.data(), sm.data(), zt.data(), k, t.data(), T, V, rows.data());
    oracle_lse_merge(lparts.data(), k, T, lse.data());
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      oracle_fljsd_terms_shard_bf16(xb.data(), Wb.data() + v0 * H, xb2.data(), Wb2.data() + v0 * H, T, H, w1, 0.3,
                                    1.5, lse.data(), terms.data() + j * T, threads);
    }
    oracle_jsd_merge(terms.data(), k, T, keep.data(), rows.data());
    oracle_jsd_merge(terms.data(), k, T, nullptr, rows.data());
    // the fused JSD's shard backward: KL shares, then each shard's gradient
    std::vector<double> klsum(T, 0.0), klj(T);
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      oracle_fljsd_kl_shard_bf16(xb.data(), Wb.data() + v0 * H, xb2.data(), Wb2.data() + v0 * H, T, H, w1, 0.3, 1.5,
                                 lse.data(), klj.data(), threads);
      for (int64_t i = 0; i < T; ++i) klsum[i] += klj[i];
    }
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      oracle_fljsd_grad_shard_bf16(xb.data(), Wb.data() + v0 * H, xb2.data(), Wb2.data() + v0 * H, T, H, w1, 0.3,
                                   1.5, j == 0 ? keep.data() : nullptr, lse.data(), klsum.data(), 2.0, dx.data(),
                                   dW.data());
    }
    // the fused CE's shard backward, from the gathered partials' normalisers
    std::vector<double> glse(T);
    oracle_ce_partials_lse(m.data(), sm.data(), k, T, glse.data());
    for (int64_t j = 0; j < k; ++j) {
      const int64_t v0 = V * j / k, w1 = V * (j + 1) / k - v0;
      oracle_flce_grad_shard_bf16(xb.data(), Wb.data() + v0 * H, t.data(), T, H, w1, v0, V, glse.data(), 1.5,
                                  dx.data(), dW.data());
    }
  }
  if (T % 2 == 0) {
    const int64_t B = 2, S = T / 2;
    oracle_cpo_combine(rows2.data(), B, S, 0.1, 1.0, lp.data(), w.data());
    oracle_cpo_f64(xd.data(), Wd.data(), t.data(), B, S, H, V, 0.5, 1.3, rows.data(), lp.data());
    oracle_cpo_bf16(xb.data(), Wb.data(), t.data(), B, S, H, V, 0.1, 0.0, rows.data(), lp.data(), threads);
    oracle_cpo_grad_f64(xd.data(), Wd.data(), t.data(), B, S, H, V, 0.7, 1.0, 1.5, dx.data(), dW.data());
    oracle_cpo_grad_bf16(xb.data(), Wb.data(), t.data(), B, S, H, V, 0.1, 1.0, 1.0, dx.data(), dW.data());
  }
}

}  // namespace

int main() {
  const uint32_t ctr[4] = {0, 0, 0, 0}, key[2] = {0, 0};
  uint32_t out[4];
  gen_philox4x32_10(ctr, key, out);
  // ragged shapes: V = 1, odd T/H/V, a shape larger than the thread count
  const int64_t shapes[][3] = {{1, 1, 1}, {2, 3, 1}, {3, 5, 7}, {6, 8, 13}, {10, 16, 33}, {17, 9, 64}};
  for (const auto& s : shapes)
    for (int threads : {1, 4}) run_shape(s[0], s[1], s[2], threads);
  std::printf("sanitize driver: ok\n");
  return 0;
}
