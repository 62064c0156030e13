// Seeded synthetic input generator shared by the GPU tests, the bench and the
// oracle tests.  It holds none of the loss arithmetic: it only turns
// (seed, stream, element index) into the bytes of an input tensor.
//
// Counter-based so any slice of any tensor can be produced independently and
// in parallel with identical results (a full-size tensor on the device and a
// handful of its rows on the host agree bit for bit):
//   * Philox4x32-10, Salmon, Moraes, Dror & Shaw, "Parallel random numbers:
//     as easy as 1, 2, 3", SC'11: key = (low 32 bits of seed, stream id),
//     counter = (block index low, block index high, high 32 bits of seed, 0).
//   * Normals: Box-Muller in double precision.  Block j gives elements 2j
//     (cosine branch) and 2j+1 (sine branch); u1 in (0,1] from words 0-1,
//     u2 in [0,1) from words 2-3, 53 bits each.  The normal is multiplied by
//     sigma in double, rounded to nearest-even to fp32, and for bf16 outputs
//     rounded once more, nearest-even, from fp32 to bf16.
//   * Targets: element 2j takes the 64-bit word (w1:w0) of block j, element
//     2j+1 takes (w3:w2); the value in [0, V) is the high half of the 128-bit
//     product word*V (Lemire's multiply-shift; bias below V/2^64).
//
// Portable C++17 only (no intrinsics), so that x86-64 and aarch64 hosts make
// the same bytes.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Block { uint32_t w[4]; };

inline void mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = static_cast<uint64_t>(a) * static_cast<uint64_t>(b);
  *hi = static_cast<uint32_t>(p >> 32);
  *lo = static_cast<uint32_t>(p);
}

inline Block philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                           uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo32(M0, c0, &hi0, &lo0);
    mulhilo32(M1, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0; k1 += W1;
  }
  return Block{{c0, c1, c2, c3}};
}

inline Block block_at(uint64_t seed, uint32_t stream, uint64_t j) {
  return philox4x32_10(static_cast<uint32_t>(j), static_cast<uint32_t>(j >> 32),
                       static_cast<uint32_t>(seed >> 32), 0u,
                       static_cast<uint32_t>(seed), stream);
}

// 53-bit uniform from a 64-bit word.
inline double u53(uint64_t w) { return static_cast<double>(w >> 11) * 0x1.0p-53; }

// Both normals of block j (elements 2j and 2j+1).
inline void normal_pair(uint64_t seed, uint32_t stream, uint64_t j, double* n0, double* n1) {
  Block b = block_at(seed, stream, j);
  uint64_t a = (static_cast<uint64_t>(b.w[1]) << 32) | b.w[0];
  uint64_t c = (static_cast<uint64_t>(b.w[3]) << 32) | b.w[2];
  double u1 = 1.0 - u53(a);             // (0, 1]
  double u2 = u53(c);                   // [0, 1)
  double r = std::sqrt(-2.0 * std::log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  *n0 = r * std::cos(th);
  *n1 = r * std::sin(th);
}

// Calls emit(k, value) for k in [lo, hi), value = normal of element offset+k.
template <class Emit>
void normals_range(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t lo, uint64_t hi,
                   Emit emit) {
  uint64_t k = lo;
  while (k < hi) {
    uint64_t e = offset + k;
    double n0, n1;
    normal_pair(seed, stream, e >> 1, &n0, &n1);
    if (e & 1) { emit(k, n1); k += 1; continue; }
    emit(k, n0);
    if (k + 1 < hi) emit(k + 1, n1);
    k += 2;
  }
}

// fp32 -> bf16, round to nearest even (NaN kept quiet).
inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return static_cast<uint16_t>((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

template <class F>
void parallel_for(uint64_t n, int threads, F f) {
  if (threads <= 1 || n < 65536) { f(0, n); return; }
  std::vector<std::thread> pool;
  uint64_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    uint64_t lo = t * chunk, hi = lo + chunk < n ? lo + chunk : n;
    if (lo >= hi) break;
    pool.emplace_back([=] { f(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Raw Philox4x32-10 block, for known-answer tests.
void gen_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  Block b = philox4x32_10(ctr[0], ctr[1], ctr[2], ctr[3], key[0], key[1]);
  for (int k = 0; k < 4; ++k) out[k] = b.w[k];
}

// Elements [offset, offset+n) of the N(0, sigma^2) fp64 stream (before rounding).
void gen_normal_f64(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n,
                    double sigma, double* out, int threads) {
  parallel_for(n, threads, [&](uint64_t lo, uint64_t hi) {
    normals_range(seed, stream, offset, lo, hi, [&](uint64_t k, double v) { out[k] = sigma * v; });
  });
}

void gen_normal_f32(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n,
                    double sigma, float* out, int threads) {
  parallel_for(n, threads, [&](uint64_t lo, uint64_t hi) {
    normals_range(seed, stream, offset, lo, hi,
                  [&](uint64_t k, double v) { out[k] = static_cast<float>(sigma * v); });
  });
}

void gen_normal_bf16(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n,
                     double sigma, uint16_t* out, int threads) {
  parallel_for(n, threads, [&](uint64_t lo, uint64_t hi) {
    normals_range(seed, stream, offset, lo, hi, [&](uint64_t k, double v) {
      out[k] = f32_to_bf16_rne(static_cast<float>(sigma * v));
    });
  });
}

void gen_targets(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n,
                 int64_t V, int64_t* out, int threads) {
  parallel_for(n, threads, [&](uint64_t lo, uint64_t hi) {
    for (uint64_t i = lo; i < hi; ++i) {
      uint64_t e = offset + i;
      Block b = block_at(seed, stream, e >> 1);
      uint64_t w = (e & 1) ? ((static_cast<uint64_t>(b.w[3]) << 32) | b.w[2])
                           : ((static_cast<uint64_t>(b.w[1]) << 32) | b.w[0]);
      unsigned __int128 p = static_cast<unsigned __int128>(w) * static_cast<uint64_t>(V);
      out[i] = static_cast<int64_t>(static_cast<uint64_t>(p >> 64));
    }
  });
}

}  // extern "C"
