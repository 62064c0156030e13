// C ABI entry points (include/lmho.h): argument checks, workspace carve-up,
// TMA tensor maps and kernel selection.  Nothing here allocates or
// synchronises except lmho_ws_status, which is documented to.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/lmho.h"
#include "lmho_internal.h"
#include "ptx.cuh"
#include "transfer.h"

namespace lmho {
namespace {

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

constexpr size_t kAlign = 256;
inline size_t align_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

struct DeviceInfo {
  bool checked = false;
  bool ok = false;
  int num_sms = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// Compute capability 10.3 (sm_103) is the only target the kernels are built for.
int current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LMHO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LMHO_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.checked = true;
  }
  if (!d.ok) return LMHO_ERR_UNSUPPORTED;
  *num_sms = d.num_sms;
  return LMHO_OK;
}

struct Range {
  uintptr_t lo, hi;
};
inline Range rng(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Each `out` range must be disjoint from every input range and from the other outputs.
int check_alias(const Range* in, int nin, const Range* out, int nout) {
  for (int i = 0; i < nout; ++i) {
    for (int j = 0; j < nin; ++j)
      if (overlap(out[i], in[j])) return LMHO_ERR_ALIAS;
    for (int j = i + 1; j < nout; ++j)
      if (overlap(out[i], out[j])) return LMHO_ERR_ALIAS;
  }
  return LMHO_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? LMHO_OK : LMHO_ERR_CUDA; }

inline Ctrl* ctrl_of(void* ws, size_t ws_bytes) {
  return reinterpret_cast<Ctrl*>(static_cast<char*>(ws) + (ws_bytes / kAlign) * kAlign - kAlign);
}

// ---------------------------------------------------------------- CE selection
// Process-wide decomposition override (lmho_set_ce_variant); initial value
// from LMHO_CE_VARIANT = warp | cta | cta512 | cluster2 | cluster4 | cluster8.
int env_ce_variant() {
  const char* s = std::getenv("LMHO_CE_VARIANT");
  if (!s) return 0;
  const char* names[] = {"warp", "cta", "cta512", "cluster2", "cluster4", "cluster8", "bulk"};
  for (int i = 0; i < 7; ++i)
    if (!std::strcmp(s, names[i])) return i + 1;
  return 0;
}
std::atomic<int> g_ce_variant{env_ce_variant()};
std::atomic<int> g_group_m{0};

// Measurement knob: LMHO_CE_BULK_RING_KB (16..200) sets the bulk ring size.
uint32_t env_bulk_ring() {
  const char* s = std::getenv("LMHO_CE_BULK_RING_KB");
  if (!s) return 0;
  const long kb = std::strtol(s, nullptr, 10);
  return (kb >= 16 && kb <= 200) ? static_cast<uint32_t>(kb) * 1024u : 0u;
}
const uint32_t g_bulk_ring = env_bulk_ring();


// Rows the bulk-copy ring can take: whole 16-byte vectors, 16-byte aligned
// start, two stages in the ring.
bool bulk_ok(const void* base, int64_t V, size_t elt) {
  const uint64_t row_bytes = static_cast<uint64_t>(V) * elt;
  return (reinterpret_cast<uintptr_t>(base) & 15u) == 0 && row_bytes % 16 == 0 && row_bytes <= kCeBulkMaxRow;
}

}  // namespace

namespace {
// Memory the GPU owns (device or managed), as opposed to host memory mapped
// into the address space (pinned, registered, or pageable through ATS).
bool device_resident(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}
}  // namespace

CeConfig choose_ce(const void* base, int64_t rows, int64_t V, size_t elt, int num_sms) {
  CeConfig c{kCeCta, 256, 1};
  c.num_sms = num_sms;
  c.timeout_ns = g_timeout_ns.load();
  c.bulk_ring_bytes = g_bulk_ring;
  const int64_t row_bytes = V * static_cast<int64_t>(elt);
  switch (g_ce_variant.load()) {
    case 1: c.variant = kCeWarp; return c;
    case 2: return c;
    case 3: c.threads = 512; return c;
    case 4: c.variant = kCeCluster; c.cluster = 2; return c;
    case 5: c.variant = kCeCluster; c.cluster = 4; return c;
    case 6: c.variant = kCeCluster; c.cluster = 8; return c;
    case 7:
      // the ring copies rows with cp.async.bulk: device-resident logits only;
      // otherwise (e.g. pinned host memory) the automatic choice below
      if (bulk_ok(base, V, elt) && device_resident(base)) {
        c.variant = kCeBulk;
        return c;
      }
      break;
    default: break;
  }
  // Measured on GB300 (flat fp32 [16384, V], Megatron bf16 [2048, 4, V],
  // calls back to back over inputs larger than L2): rows of at most 32 KB
  // stream fastest through warp-per-row loads (fp32 V = 4096: 43.3 us against
  // 46.9 for the bulk-copy ring; V = 8192: 82.5 against 83.3); longer rows
  // through a CTA per row (fp32 V = 16384: 149 us, warp per row 155, ring 352).
  if (row_bytes <= 32 * 1024) {
    c.variant = kCeWarp;
  } else if (rows < 4 * static_cast<int64_t>(num_sms) && row_bytes >= 64 * 1024) {
    c.variant = kCeCluster;   // few long rows: split each row over a cluster
    c.cluster = 8;
  }
  return c;
}

namespace {

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? LMHO_OK : LMHO_ERR_CUDA;
}

// bf16 matrix [rows, K] (row-major, K contiguous, row stride ld >= K elements,
// ld * 2 a multiple of 16), box = 64 (K) x box_rows, 128-byte swizzle; reads
// past K or past the last row are zero-filled.
int tmap_bf16_ld(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t ld, uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LMHO_OK : LMHO_ERR_CUDA;
}
int tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t H, uint32_t box_rows) {
  return tmap_bf16_ld(m, base, rows, H, H, box_rows);
}

// bf16 matrix [k_rows, mn] (row-major, MN contiguous, row stride ld >= mn
// elements, ld * 2 a multiple of 16) read MN-major: box = 64 (MN) x 64 (K),
// 128-byte swizzle; reads past either edge are zero-filled.
// `tile_mn` = the MN extent of the operand's tile (a multiple of kMnChunk).
// With mn_chunked(mn) the map is 3-D: (64 contiguous elements, K rows at ld,
// chunks 128 bytes apart), box (64, kBK, tile_mn / 64); the chunks land
// kBK * 128 bytes apart in shared memory, as separate 2-D boxes would.  Every
// chunk index below mn / 64 addresses only elements below mn.
int tmap_bf16_mn(CUtensorMap* m, const void* base, int64_t k_rows, int64_t mn, int64_t ld, int tile_mn) {
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (mn_chunked(mn)) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kMnChunk), static_cast<cuuint64_t>(k_rows),
                          static_cast<cuuint64_t>(mn / kMnChunk)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(kMnChunk) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kMnChunk), static_cast<cuuint32_t>(kBK),
                         static_cast<cuuint32_t>(tile_mn / kMnChunk)};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(mn), static_cast<cuuint64_t>(k_rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kMnChunk), static_cast<cuuint32_t>(kBK)};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? LMHO_OK : LMHO_ERR_CUDA;
}

// `group` = the default raster group of the pass (lmho_set_raster_group overrides it).
FusedGeometry geometry(int64_t T, int64_t H, int64_t V, int bn, int group = kGroupSingle) {
  FusedGeometry g{};
  g.T = T;
  g.H = H;
  g.V = V;
  g.num_m = (T + kBM - 1) / kBM;
  g.num_n = (V + bn - 1) / bn;
  const int over = g_group_m.load();
  const int64_t want = over > 0 ? over : group;
  g.group_m = static_cast<int>(g.num_m < want ? g.num_m : want);
  g.group_store = over > 0 ? over : kGroupStore;
  return g;
}

int check_fused_common(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || H <= 0 || V <= 0) return LMHO_ERR_INVALID_ARG;
  if (H % 8 != 0) return LMHO_ERR_UNSUPPORTED;  // TMA row stride must be a multiple of 16 bytes
  if (T > (int64_t(1) << 31) || V > (int64_t(1) << 31)) return LMHO_ERR_INVALID_ARG;
  return LMHO_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// The measurement hook is per host thread (each thread's own events).
thread_local cudaEvent_t t_events[16];
thread_local int t_nevents = 0;

}  // namespace

void launch_mark(int i, cudaStream_t st) {
  if (i < t_nevents && t_events[i]) cudaEventRecord(t_events[i], st);
}

// ---------------------------------------------------------------- workspace layouts
size_t flce_ws_bytes(int64_t T, int64_t H, int64_t V) {
  (void)H;
  const int64_t num_n = (V + kBN_CE - 1) / kBN_CE;
  return align_up(4 * T) + 3 * align_up(4 * num_n * T) + kAlign;
}
FusedWs flce_ws_carve(void* ws, size_t ws_bytes, int64_t T, int64_t V) {
  const int64_t num_n = (V + kBN_CE - 1) / kBN_CE;
  char* p = static_cast<char*>(ws);
  FusedWs w{};
  w.row_out = reinterpret_cast<float*>(p);
  p += align_up(4 * T);
  w.part0 = reinterpret_cast<float*>(p);
  p += align_up(4 * num_n * T);
  w.part1 = reinterpret_cast<float*>(p);
  p += align_up(4 * num_n * T);
  w.part2 = reinterpret_cast<float*>(p);
  w.ctrl = ctrl_of(ws, ws_bytes);
  return w;
}
// Fused linear + CE backward: the forward's workspace, then the log-sum-exp of
// every row, dZ (bf16, row stride padded to whole 256-column tiles) and the
// fp32 K slices of a split gradient product (sized for the larger of dx and dW
// where either can split).
namespace {
struct BwdLayout {
  int64_t ld_dz;
  size_t off_lse, off_dz, off_split, split_bytes, end;
};
// `base` = the forward's workspace bytes (its carve-up comes first, with its
// control block moved to the very end).
BwdLayout bwd_layout(int64_t T, int64_t H, int64_t V, size_t base) {
  BwdLayout b{};
  b.ld_dz = (V + kBN_CE - 1) / kBN_CE * kBN_CE;
  size_t o = base;
  b.off_lse = o;
  o += align_up(4 * static_cast<size_t>(T));
  b.off_dz = o;
  o += align_up(2 * static_cast<size_t>(T) * b.ld_dz);
  const size_t rx = k_split_reserve_bytes(T, H), rw = k_split_reserve_bytes(V, H);
  b.split_bytes = rx > rw ? rx : rw;
  b.off_split = o;
  o += align_up(b.split_bytes);
  b.end = o + kAlign;  // the control block stays the last 256 bytes
  return b;
}
}  // namespace

size_t flce_bwd_ws_bytes(int64_t T, int64_t H, int64_t V) {
  return bwd_layout(T, H, V, flce_ws_bytes(T, H, V)).end;
}

namespace {
FlceBwdWs bwd_carve(void* ws, const BwdLayout& b) {
  char* p = static_cast<char*>(ws);
  FlceBwdWs w{};
  w.lse = reinterpret_cast<float*>(p + b.off_lse);
  w.dz = reinterpret_cast<uint16_t*>(p + b.off_dz);
  w.split = b.split_bytes ? reinterpret_cast<float*>(p + b.off_split) : nullptr;
  w.ld_dz = b.ld_dz;
  return w;
}
}  // namespace

FlceBwdWs flce_bwd_ws_carve(void* ws, int64_t T, int64_t H, int64_t V) {
  return bwd_carve(ws, bwd_layout(T, H, V, flce_ws_bytes(T, H, V)));
}

// CPO: the fused CE's workspace, then lp [B], sig [B/2] and one slot for the
// token mean; the backward adds the flce backward buffers and row weights [T].
namespace {
struct CpoLayout {
  size_t off_lp, off_sig, off_mean, end;  // end includes a control-block slot
};
CpoLayout cpo_layout(int64_t B, int64_t S, int64_t H, int64_t V) {
  CpoLayout c{};
  size_t o = flce_ws_bytes(B * S, H, V);
  c.off_lp = o;
  o += align_up(4 * static_cast<size_t>(B));
  c.off_sig = o;
  o += align_up(4 * static_cast<size_t>(B));
  c.off_mean = o;
  o += kAlign;
  c.end = o + kAlign;
  return c;
}
size_t cpo_bwd_ws_bytes(int64_t B, int64_t S, int64_t H, int64_t V) {
  return bwd_layout(B * S, H, V, cpo_layout(B, S, H, V).end).end + align_up(4 * static_cast<size_t>(B * S));
}
}  // namespace

// JSD backward: the JSD forward's workspace, then the same backward buffers
// (the per-row slot holds KL(P || M)), then one float for 1 / kept count.
size_t fljsd_bwd_ws_bytes(int64_t T, int64_t H, int64_t V) {
  return bwd_layout(T, H, V, fljsd_ws_bytes(T, H, V)).end + kAlign;
}

// Partials: the log-sum-exp pass writes (max, sum) per (head, 256-wide vocab
// tile); the divergence pass writes one sum per (kBN_JSD-wide vocab tile,
// epilogue column slice).  part0 serves both passes.
size_t fljsd_ws_bytes(int64_t T, int64_t H, int64_t V) {
  (void)H;
  const int64_t n256 = (V + kBN_CE - 1) / kBN_CE;
  const int64_t njsd = (V + kBN_JSD - 1) / kBN_JSD * kJsdColSplit;
  const int64_t p0 = (2 * n256 > njsd ? 2 * n256 : njsd) * T;
  // part0 and part1 both hold either pass's partials: (max, sum) of the
  // log-sum-exp pass, or the divergence and KL(P || M) sums of the JSD pass
  return align_up(4 * T) + 2 * align_up(4 * p0) + align_up(4 * 2 * T) + kAlign;
}
FusedWs fljsd_ws_carve(void* ws, size_t ws_bytes, int64_t T, int64_t V) {
  const int64_t n256 = (V + kBN_CE - 1) / kBN_CE;
  const int64_t njsd = (V + kBN_JSD - 1) / kBN_JSD * kJsdColSplit;
  const int64_t p0 = (2 * n256 > njsd ? 2 * n256 : njsd) * T;
  char* p = static_cast<char*>(ws);
  FusedWs w{};
  w.row_out = reinterpret_cast<float*>(p);
  p += align_up(4 * T);
  w.part0 = reinterpret_cast<float*>(p);
  p += align_up(4 * p0);
  w.part1 = reinterpret_cast<float*>(p);
  p += align_up(4 * p0);
  w.lse = reinterpret_cast<float*>(p);
  w.ctrl = ctrl_of(ws, ws_bytes);
  return w;
}

}  // namespace lmho

using namespace lmho;

extern "C" {

const char* lmho_strerror(int status) {
  switch (status) {
    case LMHO_OK: return "ok";
    case LMHO_ERR_INVALID_ARG: return "invalid argument (null pointer, size <= 0 or out of range)";
    case LMHO_ERR_ALIAS: return "an output or workspace range overlaps an input or another output";
    case LMHO_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case LMHO_ERR_UNSUPPORTED: return "unsupported: device is not compute capability 10.3, or H % 8 != 0";
    case LMHO_ERR_CUDA: return "a CUDA runtime call failed";
    case LMHO_ERR_TIMEOUT: return "a bounded in-kernel wait timed out";
    default: return "unknown status";
  }
}

int lmho_version(void) { return 200; }

void lmho_set_launch_events(void* const* events, int n) {
  t_nevents = 0;
  if (!events || n <= 0) return;
  if (n > 16) n = 16;
  for (int k = 0; k < n; ++k) t_events[k] = static_cast<cudaEvent_t>(events[k]);
  t_nevents = n;
}

int lmho_set_raster_group(int group_m) {
  if (group_m < 0 || group_m > 1024) return LMHO_ERR_INVALID_ARG;
  g_group_m.store(group_m);
  return LMHO_OK;
}

int lmho_set_ce_variant(int variant) {
  if (variant < 0 || variant > 7) return LMHO_ERR_INVALID_ARG;
  g_ce_variant.store(variant);
  return LMHO_OK;
}

void lmho_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

size_t ce_workspace_bytes(int64_t T, int64_t V) {
  (void)V;
  if (T <= 0) return kAlign;
  return align_up(4 * static_cast<size_t>(T)) + kAlign;
}

int ce_fwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V, float* loss, void* ws,
               size_t ws_bytes, void* stream) {
  if (!logits || !target || !loss || !ws) return LMHO_ERR_INVALID_ARG;
  if (T <= 0 || V <= 0 || T > (int64_t(1) << 31) - 1) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < ce_workspace_bytes(T, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[2] = {rng(logits, 4 * static_cast<size_t>(T) * V), rng(target, 8 * static_cast<size_t>(T))};
  const Range out[2] = {rng(loss, 4), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 2, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  const CeConfig cfg = choose_ce(logits, T, V, 4, sms);
  return cuda_status(launch_ce_f32(logits, target, T, V, loss, static_cast<float*>(ws), ctrl_of(ws, ws_bytes), cfg,
                                   static_cast<cudaStream_t>(stream)));
}

int ce_fwd_sbv_bf16(const uint16_t* logits, const int64_t* target, int64_t S, int64_t B, int64_t V, float* loss,
                    void* stream) {
  if (!logits || !target || !loss) return LMHO_ERR_INVALID_ARG;
  if (S <= 0 || B <= 0 || V <= 0) return LMHO_ERR_INVALID_ARG;
  const int64_t rows = S * B;
  if (rows > (int64_t(1) << 31) - 1) return LMHO_ERR_INVALID_ARG;
  const Range in[2] = {rng(logits, 2 * static_cast<size_t>(rows) * V), rng(target, 8 * static_cast<size_t>(rows))};
  const Range out[1] = {rng(loss, 4 * static_cast<size_t>(rows))};
  if (int a = check_alias(in, 2, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  const CeConfig cfg = choose_ce(logits, rows, V, 2, sms);
  return cuda_status(launch_ce_bf16_rows(logits, target, rows, V, loss, cfg, static_cast<cudaStream_t>(stream)));
}

int ce_partials_sbv_bf16(const uint16_t* logits_local, const int64_t* target, int64_t S, int64_t B,
                         int64_t V_local, int64_t vocab_start, float* partials, void* stream) {
  if (!logits_local || !target || !partials) return LMHO_ERR_INVALID_ARG;
  if (S <= 0 || B <= 0 || V_local <= 0 || vocab_start < 0) return LMHO_ERR_INVALID_ARG;
  const int64_t rows = S * B;
  if (rows > (int64_t(1) << 31) - 1 || vocab_start > (int64_t(1) << 62)) return LMHO_ERR_INVALID_ARG;
  const Range in[2] = {rng(logits_local, 2 * static_cast<size_t>(rows) * V_local),
                       rng(target, 8 * static_cast<size_t>(rows))};
  const Range out[1] = {rng(partials, 12 * static_cast<size_t>(rows))};
  if (int a = check_alias(in, 2, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  CeConfig cfg = choose_ce(logits_local, rows, V_local, 2, sms);
  return cuda_status(launch_ce_partials_bf16(logits_local, target, rows, V_local, vocab_start, partials, cfg,
                                             static_cast<cudaStream_t>(stream)));
}

int ce_partials_f32(const float* logits_local, const int64_t* target, int64_t T, int64_t V_local,
                    int64_t vocab_start, float* partials, void* stream) {
  if (!logits_local || !target || !partials) return LMHO_ERR_INVALID_ARG;
  if (T <= 0 || V_local <= 0 || vocab_start < 0) return LMHO_ERR_INVALID_ARG;
  if (T > (int64_t(1) << 31) - 1 || vocab_start > (int64_t(1) << 62)) return LMHO_ERR_INVALID_ARG;
  const Range in[2] = {rng(logits_local, 4 * static_cast<size_t>(T) * V_local), rng(target, 8 * static_cast<size_t>(T))};
  const Range out[1] = {rng(partials, 12 * static_cast<size_t>(T))};
  if (int a = check_alias(in, 2, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  const CeConfig cfg = choose_ce(logits_local, T, V_local, 4, sms);
  return cuda_status(launch_ce_partials_f32(logits_local, target, T, V_local, vocab_start, partials, cfg,
                                            static_cast<cudaStream_t>(stream)));
}

int ce_merge_partials(const float* partials, int64_t shards, const int64_t* target, int64_t S, int64_t B, int64_t V,
                      float* loss, void* stream) {
  if (!partials || !target || !loss) return LMHO_ERR_INVALID_ARG;
  if (shards <= 0 || S <= 0 || B <= 0 || V <= 0) return LMHO_ERR_INVALID_ARG;
  const int64_t rows = S * B;
  if (rows > (int64_t(1) << 31) - 1 || shards > (int64_t(1) << 20)) return LMHO_ERR_INVALID_ARG;
  const Range in[2] = {rng(partials, 12 * static_cast<size_t>(rows) * static_cast<size_t>(shards)),
                       rng(target, 8 * static_cast<size_t>(rows))};
  const Range out[1] = {rng(loss, 4 * static_cast<size_t>(rows))};
  if (int a = check_alias(in, 2, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_ce_merge(partials, shards, target, rows, V, loss, sms, static_cast<cudaStream_t>(stream)));
}

int ce_fwd_bwd_f32(const float* logits, const int64_t* target, int64_t T, int64_t V, float grad_scale, float* loss,
                   float* dlogits, void* ws, size_t ws_bytes, void* stream) {
  if (!logits || !target || !loss || !dlogits || !ws) return LMHO_ERR_INVALID_ARG;
  if (T <= 0 || V <= 0 || T > (int64_t(1) << 31) / 8) return LMHO_ERR_INVALID_ARG;
  if (!std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < ce_workspace_bytes(T, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const size_t zb = 4 * static_cast<size_t>(T) * V;
  const Range in[2] = {rng(logits, zb), rng(target, 8 * static_cast<size_t>(T))};
  const Range out[3] = {rng(loss, 4), rng(dlogits, zb), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 2, out, 3)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_ce_fwd_bwd_f32(logits, target, T, V, grad_scale / static_cast<float>(T), loss,
                                           static_cast<float*>(ws), dlogits, ctrl_of(ws, ws_bytes),
                                           g_timeout_ns.load(), static_cast<cudaStream_t>(stream)));
}

int ce_fwd_bwd_sbv_bf16(const uint16_t* logits, const int64_t* target, int64_t S, int64_t B, int64_t V,
                        const float* dloss, float grad_scale, float* loss, uint16_t* dlogits, void* stream) {
  if (!logits || !target || !loss || !dlogits) return LMHO_ERR_INVALID_ARG;
  if (S <= 0 || B <= 0 || V <= 0) return LMHO_ERR_INVALID_ARG;
  const int64_t rows = S * B;
  if (rows > (int64_t(1) << 31) / 8) return LMHO_ERR_INVALID_ARG;
  if (!std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  const size_t zb = 2 * static_cast<size_t>(rows) * V;
  const Range in[3] = {rng(logits, zb), rng(target, 8 * static_cast<size_t>(rows)),
                       rng(dloss, dloss ? 4 * static_cast<size_t>(rows) : 0)};
  const Range out[2] = {rng(loss, 4 * static_cast<size_t>(rows)), rng(dlogits, zb)};
  if (int a = check_alias(in, 3, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_ce_fwd_bwd_bf16_rows(logits, target, rows, V, dloss, grad_scale, loss, dlogits,
                                                 g_timeout_ns.load(), static_cast<cudaStream_t>(stream)));
}

size_t flce_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || V <= 0) return kAlign;
  return flce_ws_bytes(T, H, V);
}

int flce_fwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T, int64_t H, int64_t V,
                  float* loss, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !W || !target || !loss || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V)) return c;
  if (!aligned16(x) || !aligned16(W)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < flce_ws_bytes(T, H, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[3] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W, 2 * static_cast<size_t>(V) * H),
                       rng(target, 8 * static_cast<size_t>(T))};
  const Range out[2] = {rng(loss, 4), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 3, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap tx, tw;
  if (tmap_bf16(&tx, x, T, H, kBM) || tmap_bf16(&tw, W, V, H, kBoxBFwd)) return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V, kBN_CE);
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce(tx, tw, target, g, loss, w, L));
}

size_t flce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || V <= 0 || H <= 0) return kAlign;
  return flce_bwd_ws_bytes(T, H, V);
}

int flce_fwd_bwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t T, int64_t H, int64_t V,
                      float grad_scale, float* loss, float* dx, float* dW, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !W || !target || !loss || !dx || !dW || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V)) return c;
  if (!std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W) || !aligned16(dx) || !aligned16(dW)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < flce_bwd_ws_bytes(T, H, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[3] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W, 2 * static_cast<size_t>(V) * H),
                       rng(target, 8 * static_cast<size_t>(T))};
  const Range out[4] = {rng(loss, 4), rng(dx, 4 * static_cast<size_t>(T) * H), rng(dW, 4 * static_cast<size_t>(V) * H),
                        rng(ws, ws_bytes)};
  if (int a = check_alias(in, 3, out, 4)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V);
  const FlceBwdWs bw = flce_bwd_ws_carve(ws, T, H, V);
  FlceBwdMaps m;
  if (tmap_bf16(&m.x, x, T, H, kBM) || tmap_bf16(&m.w, W, V, H, kBoxBFwd) ||
      tmap_bf16_ld(&m.dz, bw.dz, T, V, bw.ld_dz, kBM) || tmap_bf16_mn(&m.w_mn, W, V, H, H, kBoxBGrad) ||
      tmap_bf16_mn(&m.dz_mn, bw.dz, T, V, bw.ld_dz, kBM) || tmap_bf16_mn(&m.x_mn, x, T, H, H, kBoxBGrad))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V, kBN_CE);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce_fwd_bwd(m, target, g, grad_scale, loss, dx, dW, w, bw, L));
}

size_t fljsd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || V <= 0) return kAlign;
  return fljsd_ws_bytes(T, H, V);
}

namespace {
int fljsd_impl(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T, int64_t H,
               int64_t V, float beta, float temperature, const uint8_t* keep, float* loss, void* ws, size_t ws_bytes,
               void* stream) {
  if (!xs || !Ws || !xt || !Wt || !loss || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V)) return c;
  if (!(beta > 0.f && beta < 1.f)) return LMHO_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(1.f / temperature < INFINITY)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16(Ws) || !aligned16(xt) || !aligned16(Wt)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < fljsd_ws_bytes(T, H, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const size_t xb = 2 * static_cast<size_t>(T) * H, wb = 2 * static_cast<size_t>(V) * H;
  const Range in[5] = {rng(xs, xb), rng(Ws, wb), rng(xt, xb), rng(Wt, wb), rng(keep, keep ? static_cast<size_t>(T) : 0)};
  const Range out[2] = {rng(loss, 4), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 5, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap txs, txt, tws256, twt256, twsj, twtj;
  if (tmap_bf16(&txs, xs, T, H, kBM) || tmap_bf16(&txt, xt, T, H, kBM) || tmap_bf16(&tws256, Ws, V, H, kBoxBFwd) ||
      tmap_bf16(&twt256, Wt, V, H, kBoxBFwd) || tmap_bf16(&twsj, Ws, V, H, kBN_JSD) ||
      tmap_bf16(&twtj, Wt, V, H, kBN_JSD))
    return LMHO_ERR_CUDA;
  const FusedGeometry g1 = geometry(T, H, V, kBN_CE), g2 = geometry(T, H, V, kBN_JSD, kGroupTwoHead);
  const FusedWs w = fljsd_ws_carve(ws, ws_bytes, T, V);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(
      launch_fljsd(txs, tws256, txt, twt256, twsj, twtj, g1, g2, beta, 1.f / temperature, keep, loss, w, L));
}
}  // namespace

int fljsd_fwd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T,
                   int64_t H, int64_t V, float beta, float* loss, void* ws, size_t ws_bytes, void* stream) {
  return fljsd_impl(xs, Ws, xt, Wt, T, H, V, beta, 1.f, nullptr, loss, ws, ws_bytes, stream);
}

int fljsd_fwd_bf16_ex(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T,
                      int64_t H, int64_t V, float beta, float temperature, const uint8_t* keep, float* loss, void* ws,
                      size_t ws_bytes, void* stream) {
  return fljsd_impl(xs, Ws, xt, Wt, T, H, V, beta, temperature, keep, loss, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- vocab-parallel fused losses
int flce_partials_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target, int64_t T, int64_t H,
                       int64_t V_local, int64_t vocab_start, float* partials, void* ws, size_t ws_bytes,
                       void* stream) {
  if (!x || !W_local || !target || !partials || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V_local)) return c;
  if (vocab_start < 0 || vocab_start > (int64_t(1) << 62)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_local)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < flce_ws_bytes(T, H, V_local) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[3] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W_local, 2 * static_cast<size_t>(V_local) * H),
                       rng(target, 8 * static_cast<size_t>(T))};
  const Range out[2] = {rng(partials, 12 * static_cast<size_t>(T)), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 3, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap tx, tw;
  if (tmap_bf16(&tx, x, T, H, kBM) || tmap_bf16(&tw, W_local, V_local, H, kBoxBFwd)) return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V_local, kBN_CE);
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V_local);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce_partials(tx, tw, target, vocab_start, g, partials, w, L));
}

namespace {
int flce_shard_bwd_impl(const uint16_t* x, const uint16_t* W_local, const int64_t* target, const float* partials,
                        int64_t shards, int64_t T, int64_t H, int64_t V_local, int64_t vocab_start, int64_t V,
                        const float* row_w, float grad_scale, float* dx_partial, float* dW_local, void* ws,
                        size_t ws_bytes, void* stream) {
  if (!x || !W_local || !target || !partials || !dx_partial || !dW_local || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V_local)) return c;
  if (shards <= 0 || shards > (int64_t(1) << 20) || V > (int64_t(1) << 31) || vocab_start < 0 || V < V_local ||
      vocab_start > V - V_local)
    return LMHO_ERR_INVALID_ARG;
  if (!std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_local) || !aligned16(dx_partial) || !aligned16(dW_local))
    return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < flce_bwd_ws_bytes(T, H, V_local) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[5] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W_local, 2 * static_cast<size_t>(V_local) * H),
                       rng(target, 8 * static_cast<size_t>(T)),
                       rng(partials, 12 * static_cast<size_t>(T) * static_cast<size_t>(shards)),
                       rng(row_w, row_w ? 4 * static_cast<size_t>(T) : 0)};
  const Range out[3] = {rng(dx_partial, 4 * static_cast<size_t>(T) * H),
                        rng(dW_local, 4 * static_cast<size_t>(V_local) * H), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 5, out, 3)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V_local);
  const FlceBwdWs bw = flce_bwd_ws_carve(ws, T, H, V_local);
  FlceBwdMaps m;
  if (tmap_bf16(&m.x, x, T, H, kBM) || tmap_bf16(&m.w, W_local, V_local, H, kBoxBFwd) ||
      tmap_bf16_ld(&m.dz, bw.dz, T, V_local, bw.ld_dz, kBM) || tmap_bf16_mn(&m.w_mn, W_local, V_local, H, H, kBoxBGrad) ||
      tmap_bf16_mn(&m.dz_mn, bw.dz, T, V_local, bw.ld_dz, kBM) || tmap_bf16_mn(&m.x_mn, x, T, H, H, kBoxBGrad))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V_local, kBN_CE);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce_shard_bwd(m, target, partials, shards, vocab_start, V, g, grad_scale, row_w,
                                           dx_partial, dW_local, w, bw, L));
}
}  // namespace

int flce_shard_bwd_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target, const float* partials,
                        int64_t shards, int64_t T, int64_t H, int64_t V_local, int64_t vocab_start, int64_t V,
                        float grad_scale, float* dx_partial, float* dW_local, void* ws, size_t ws_bytes,
                        void* stream) {
  return flce_shard_bwd_impl(x, W_local, target, partials, shards, T, H, V_local, vocab_start, V, nullptr,
                             grad_scale, dx_partial, dW_local, ws, ws_bytes, stream);
}

int flce_shard_bwd_rows_bf16(const uint16_t* x, const uint16_t* W_local, const int64_t* target, const float* partials,
                             int64_t shards, int64_t T, int64_t H, int64_t V_local, int64_t vocab_start, int64_t V,
                             const float* row_w, float grad_scale, float* dx_partial, float* dW_local, void* ws,
                             size_t ws_bytes, void* stream) {
  if (!row_w) return LMHO_ERR_INVALID_ARG;
  return flce_shard_bwd_impl(x, W_local, target, partials, shards, T, H, V_local, vocab_start, V, row_w,
                             grad_scale, dx_partial, dW_local, ws, ws_bytes, stream);
}

size_t cpo_combine_workspace_bytes(int64_t B) {
  if (B <= 0) return kAlign;
  return 2 * align_up(4 * static_cast<size_t>(B)) + kAlign;
}

int cpo_combine_rows(const float* rows, int64_t B, int64_t S, float beta, float alpha, float* loss, float* logps,
                     float* row_w, void* ws, size_t ws_bytes, void* stream) {
  if (!rows || !loss || !ws) return LMHO_ERR_INVALID_ARG;
  if (B < 2 || B % 2 != 0 || S <= 0 || B > (int64_t(1) << 24) || B > ((int64_t(1) << 31) - 1) / S)
    return LMHO_ERR_INVALID_ARG;
  if (!(beta > 0.f) || !std::isfinite(beta) || !(alpha >= 0.f) || !std::isfinite(alpha)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < cpo_combine_workspace_bytes(B) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const size_t T = static_cast<size_t>(B * S);
  const Range in[1] = {rng(rows, 4 * T)};
  const Range out[4] = {rng(loss, 4), rng(logps, logps ? 4 * static_cast<size_t>(B) : 0),
                        rng(row_w, row_w ? 4 * T : 0), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 1, out, 4)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  float* lp = static_cast<float*>(ws);
  float* sig = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(4 * static_cast<size_t>(B)));
  return cuda_status(launch_cpo_combine(rows, B, S, beta, alpha, loss, logps, row_w, lp, sig, ctrl_of(ws, ws_bytes),
                                        static_cast<cudaStream_t>(stream)));
}

namespace {
// Arguments shared by the two shard passes of the vocab-parallel fused JSD.
int check_jsd_shard(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T,
                    int64_t H, int64_t V_local, float temperature, void* ws, size_t ws_bytes) {
  if (!xs || !Ws || !xt || !Wt || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V_local)) return c;
  if (!(temperature > 0.f) || !(1.f / temperature < INFINITY)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16(Ws) || !aligned16(xt) || !aligned16(Wt)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < fljsd_ws_bytes(T, H, V_local) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  return LMHO_OK;
}
}  // namespace

int fljsd_lse_partials_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt, const uint16_t* Wt_local,
                            int64_t T, int64_t H, int64_t V_local, float temperature, float* lse_local, void* ws,
                            size_t ws_bytes, void* stream) {
  if (!lse_local) return LMHO_ERR_INVALID_ARG;
  if (int c = check_jsd_shard(xs, Ws_local, xt, Wt_local, T, H, V_local, temperature, ws, ws_bytes)) return c;
  const size_t xb = 2 * static_cast<size_t>(T) * H, wb = 2 * static_cast<size_t>(V_local) * H;
  const Range in[4] = {rng(xs, xb), rng(Ws_local, wb), rng(xt, xb), rng(Wt_local, wb)};
  const Range out[2] = {rng(lse_local, 8 * static_cast<size_t>(T)), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 4, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap txs, txt, tws, twt;
  if (tmap_bf16(&txs, xs, T, H, kBM) || tmap_bf16(&txt, xt, T, H, kBM) ||
      tmap_bf16(&tws, Ws_local, V_local, H, kBoxBFwd) || tmap_bf16(&twt, Wt_local, V_local, H, kBoxBFwd))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V_local, kBN_CE);
  const FusedWs w = fljsd_ws_carve(ws, ws_bytes, T, V_local);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_fljsd_lse_shard(txs, tws, txt, twt, g, 1.f / temperature, lse_local, w, L));
}

int lse_merge_partials(const float* parts, int64_t shards, int64_t T, float* lse, void* stream) {
  if (!parts || !lse) return LMHO_ERR_INVALID_ARG;
  if (shards <= 0 || shards > (int64_t(1) << 20) || T <= 0 || T > (int64_t(1) << 31) - 1)
    return LMHO_ERR_INVALID_ARG;
  const Range in[1] = {rng(parts, 8 * static_cast<size_t>(T) * static_cast<size_t>(shards))};
  const Range out[1] = {rng(lse, 8 * static_cast<size_t>(T))};
  if (int a = check_alias(in, 1, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_lse_merge(parts, shards, T, lse, sms, static_cast<cudaStream_t>(stream)));
}

int fljsd_terms_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt, const uint16_t* Wt_local,
                     const float* lse, int64_t T, int64_t H, int64_t V_local, float beta, float temperature,
                     float* terms, float* kl_local, void* ws, size_t ws_bytes, void* stream) {
  if (!lse || !terms) return LMHO_ERR_INVALID_ARG;
  if (int c = check_jsd_shard(xs, Ws_local, xt, Wt_local, T, H, V_local, temperature, ws, ws_bytes)) return c;
  if (!(beta > 0.f && beta < 1.f)) return LMHO_ERR_INVALID_ARG;
  const size_t xb = 2 * static_cast<size_t>(T) * H, wb = 2 * static_cast<size_t>(V_local) * H;
  const Range in[5] = {rng(xs, xb), rng(Ws_local, wb), rng(xt, xb), rng(Wt_local, wb),
                       rng(lse, 8 * static_cast<size_t>(T))};
  const Range out[3] = {rng(terms, 4 * static_cast<size_t>(T)), rng(ws, ws_bytes),
                        rng(kl_local, kl_local ? 4 * static_cast<size_t>(T) : 0)};
  if (int a = check_alias(in, 5, out, 3)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap txs, txt, tws, twt;
  if (tmap_bf16(&txs, xs, T, H, kBM) || tmap_bf16(&txt, xt, T, H, kBM) ||
      tmap_bf16(&tws, Ws_local, V_local, H, kBN_JSD) || tmap_bf16(&twt, Wt_local, V_local, H, kBN_JSD))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V_local, kBN_JSD, kGroupTwoHead);
  const FusedWs w = fljsd_ws_carve(ws, ws_bytes, T, V_local);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(
      launch_fljsd_terms_shard(txs, tws, txt, twt, g, lse, beta, 1.f / temperature, terms, kl_local, w, L));
}

int fljsd_shard_bwd_bf16(const uint16_t* xs, const uint16_t* Ws_local, const uint16_t* xt, const uint16_t* Wt_local,
                         const float* lse, const float* kl, const uint8_t* keep, int64_t T, int64_t H, int64_t V_local,
                         float beta, float temperature, float grad_scale, float* dxs_partial, float* dWs_local,
                         void* ws, size_t ws_bytes, void* stream) {
  if (!xs || !Ws_local || !xt || !Wt_local || !lse || !kl || !dxs_partial || !dWs_local || !ws)
    return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V_local)) return c;
  if (!(beta > 0.f && beta < 1.f)) return LMHO_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(1.f / temperature < INFINITY) || !std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16(Ws_local) || !aligned16(xt) || !aligned16(Wt_local) || !aligned16(dxs_partial) ||
      !aligned16(dWs_local))
    return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < fljsd_bwd_ws_bytes(T, H, V_local) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const size_t xb = 2 * static_cast<size_t>(T) * H, wb = 2 * static_cast<size_t>(V_local) * H;
  const Range in[7] = {rng(xs, xb), rng(Ws_local, wb), rng(xt, xb), rng(Wt_local, wb),
                       rng(lse, 8 * static_cast<size_t>(T)), rng(kl, 4 * static_cast<size_t>(T)),
                       rng(keep, keep ? static_cast<size_t>(T) : 0)};
  const Range out[3] = {rng(dxs_partial, 4 * static_cast<size_t>(T) * H),
                        rng(dWs_local, 4 * static_cast<size_t>(V_local) * H), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 7, out, 3)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  const BwdLayout lay = bwd_layout(T, H, V_local, fljsd_ws_bytes(T, H, V_local));
  const FusedWs w = fljsd_ws_carve(ws, ws_bytes, T, V_local);
  const FlceBwdWs bw = bwd_carve(ws, lay);
  float* inv_count = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.end - kAlign);
  FljsdBwdMaps m;
  if (tmap_bf16(&m.xs, xs, T, H, kBM) || tmap_bf16(&m.xt, xt, T, H, kBM) ||
      tmap_bf16(&m.wsj, Ws_local, V_local, H, kBN_JSD) || tmap_bf16(&m.wtj, Wt_local, V_local, H, kBN_JSD) ||
      tmap_bf16_ld(&m.dz, bw.dz, T, V_local, bw.ld_dz, kBM) || tmap_bf16_mn(&m.ws_mn, Ws_local, V_local, H, H, kBoxBGrad) ||
      tmap_bf16_mn(&m.dz_mn, bw.dz, T, V_local, bw.ld_dz, kBM) || tmap_bf16_mn(&m.xs_mn, xs, T, H, H, kBoxBGrad))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V_local, kBN_JSD, kGroupTwoHead);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_fljsd_shard_bwd(m, g, beta, 1.f / temperature, keep, grad_scale, lse, kl, dxs_partial,
                                            dWs_local, w, bw, inv_count, L));
}

int jsd_merge_terms(const float* terms, int64_t shards, int64_t T, const uint8_t* keep, float* rows, float* loss,
                    void* stream) {
  if (!terms || !rows || !loss) return LMHO_ERR_INVALID_ARG;
  if (shards <= 0 || shards > (int64_t(1) << 20) || T <= 0 || T > (int64_t(1) << 31) - 1)
    return LMHO_ERR_INVALID_ARG;
  if (!aligned16(rows)) return LMHO_ERR_INVALID_ARG;  // the mean reads 16-byte vectors
  const Range in[2] = {rng(terms, 4 * static_cast<size_t>(T) * static_cast<size_t>(shards)),
                       rng(keep, keep ? static_cast<size_t>(T) : 0)};
  const Range out[2] = {rng(rows, 4 * static_cast<size_t>(T)), rng(loss, 4)};
  if (int a = check_alias(in, 2, out, 2)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_jsd_merge(terms, shards, T, keep, rows, loss, sms, static_cast<cudaStream_t>(stream)));
}

int rows_mean_f32(const float* rows, int64_t n, const uint8_t* keep, float* mean, void* stream) {
  if (!rows || !mean) return LMHO_ERR_INVALID_ARG;
  if (n <= 0 || n > (int64_t(1) << 31) - 1) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(rows)) return LMHO_ERR_INVALID_ARG;
  const Range in[2] = {rng(rows, 4 * static_cast<size_t>(n)), rng(keep, keep ? static_cast<size_t>(n) : 0)};
  const Range out[1] = {rng(mean, 4)};
  if (int a = check_alias(in, 2, out, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_rows_mean(rows, n, keep, mean, static_cast<cudaStream_t>(stream)));
}

size_t fljsd_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || V <= 0 || H <= 0) return kAlign;
  return fljsd_bwd_ws_bytes(T, H, V);
}

int fljsd_fwd_bwd_bf16(const uint16_t* xs, const uint16_t* Ws, const uint16_t* xt, const uint16_t* Wt, int64_t T,
                       int64_t H, int64_t V, float beta, float temperature, const uint8_t* keep, float grad_scale,
                       float* loss, float* dxs, float* dWs, void* ws, size_t ws_bytes, void* stream) {
  if (!xs || !Ws || !xt || !Wt || !loss || !dxs || !dWs || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(T, H, V)) return c;
  if (!(beta > 0.f && beta < 1.f)) return LMHO_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(1.f / temperature < INFINITY) || !std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16(Ws) || !aligned16(xt) || !aligned16(Wt) || !aligned16(dxs) || !aligned16(dWs))
    return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < fljsd_bwd_ws_bytes(T, H, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const size_t xb = 2 * static_cast<size_t>(T) * H, wb = 2 * static_cast<size_t>(V) * H;
  const Range in[5] = {rng(xs, xb), rng(Ws, wb), rng(xt, xb), rng(Wt, wb), rng(keep, keep ? static_cast<size_t>(T) : 0)};
  const Range out[4] = {rng(loss, 4), rng(dxs, 4 * static_cast<size_t>(T) * H), rng(dWs, 4 * static_cast<size_t>(V) * H),
                        rng(ws, ws_bytes)};
  if (int a = check_alias(in, 5, out, 4)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  const BwdLayout lay = bwd_layout(T, H, V, fljsd_ws_bytes(T, H, V));
  const FusedWs w = fljsd_ws_carve(ws, ws_bytes, T, V);
  const FlceBwdWs bw = bwd_carve(ws, lay);
  float* inv_count = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.end - kAlign);
  FljsdBwdMaps m;
  if (tmap_bf16(&m.xs, xs, T, H, kBM) || tmap_bf16(&m.xt, xt, T, H, kBM) || tmap_bf16(&m.ws256, Ws, V, H, kBoxBFwd) ||
      tmap_bf16(&m.wt256, Wt, V, H, kBoxBFwd) || tmap_bf16(&m.wsj, Ws, V, H, kBN_JSD) ||
      tmap_bf16(&m.wtj, Wt, V, H, kBN_JSD) || tmap_bf16_ld(&m.dz, bw.dz, T, V, bw.ld_dz, kBM) ||
      tmap_bf16_mn(&m.ws_mn, Ws, V, H, H, kBoxBGrad) || tmap_bf16_mn(&m.dz_mn, bw.dz, T, V, bw.ld_dz, kBM) ||
      tmap_bf16_mn(&m.xs_mn, xs, T, H, H, kBoxBGrad))
    return LMHO_ERR_CUDA;
  const FusedGeometry g1 = geometry(T, H, V, kBN_CE), g2 = geometry(T, H, V, kBN_JSD, kGroupTwoHead);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_fljsd_fwd_bwd(m, g1, g2, beta, 1.f / temperature, keep, grad_scale, loss, dxs, dWs, w, bw,
                                          bw.lse, inv_count, L));
}

size_t flce_cpo_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t V) {
  if (B <= 0 || S <= 0 || H <= 0 || V <= 0) return kAlign;
  return cpo_layout(B, S, H, V).end;
}

size_t flce_cpo_bwd_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t V) {
  if (B <= 0 || S <= 0 || H <= 0 || V <= 0) return kAlign;
  return cpo_bwd_ws_bytes(B, S, H, V);
}

namespace {
int check_cpo(int64_t B, int64_t S, int64_t H, int64_t V, float beta, float alpha) {
  if (B < 2 || B % 2 != 0 || S <= 0) return LMHO_ERR_INVALID_ARG;
  if (B > (int64_t(1) << 31) / S) return LMHO_ERR_INVALID_ARG;
  if (int c = check_fused_common(B * S, H, V)) return c;
  if (!(beta > 0.f) || !std::isfinite(beta) || !(alpha >= 0.f) || !std::isfinite(alpha)) return LMHO_ERR_INVALID_ARG;
  return LMHO_OK;
}
}  // namespace

int flce_cpo_fwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B, int64_t S, int64_t H,
                      int64_t V, float beta, float alpha, float* loss, float* logps, void* ws, size_t ws_bytes,
                      void* stream) {
  if (!x || !W || !target || !loss || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_cpo(B, S, H, V, beta, alpha)) return c;
  const int64_t T = B * S;
  if (!aligned16(x) || !aligned16(W)) return LMHO_ERR_INVALID_ARG;
  const CpoLayout lay = cpo_layout(B, S, H, V);
  if (ws_bytes < lay.end || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[3] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W, 2 * static_cast<size_t>(V) * H),
                       rng(target, 8 * static_cast<size_t>(T))};
  const Range out[3] = {rng(loss, 4), rng(logps, logps ? 4 * static_cast<size_t>(B) : 0), rng(ws, ws_bytes)};
  if (int a = check_alias(in, 3, out, 3)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  CUtensorMap tx, tw;
  if (tmap_bf16(&tx, x, T, H, kBM) || tmap_bf16(&tw, W, V, H, kBoxBFwd)) return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V, kBN_CE);
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V);
  char* base = static_cast<char*>(ws);
  CpoArgs c{B, S, beta, alpha, reinterpret_cast<float*>(base + lay.off_lp), reinterpret_cast<float*>(base + lay.off_sig),
            reinterpret_cast<float*>(base + lay.off_mean), logps, nullptr};
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce_cpo(tx, tw, target, g, loss, w, c, L));
}

int flce_cpo_fwd_bwd_bf16(const uint16_t* x, const uint16_t* W, const int64_t* target, int64_t B, int64_t S,
                          int64_t H, int64_t V, float beta, float alpha, float grad_scale, float* loss, float* logps,
                          float* dx, float* dW, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !W || !target || !loss || !dx || !dW || !ws) return LMHO_ERR_INVALID_ARG;
  if (int c = check_cpo(B, S, H, V, beta, alpha)) return c;
  if (!std::isfinite(grad_scale)) return LMHO_ERR_INVALID_ARG;
  const int64_t T = B * S;
  if (!aligned16(x) || !aligned16(W) || !aligned16(dx) || !aligned16(dW)) return LMHO_ERR_INVALID_ARG;
  if (ws_bytes < cpo_bwd_ws_bytes(B, S, H, V) || !aligned256(ws)) return LMHO_ERR_WORKSPACE;
  const Range in[3] = {rng(x, 2 * static_cast<size_t>(T) * H), rng(W, 2 * static_cast<size_t>(V) * H),
                       rng(target, 8 * static_cast<size_t>(T))};
  const Range out[5] = {rng(loss, 4), rng(logps, logps ? 4 * static_cast<size_t>(B) : 0),
                        rng(dx, 4 * static_cast<size_t>(T) * H), rng(dW, 4 * static_cast<size_t>(V) * H),
                        rng(ws, ws_bytes)};
  if (int a = check_alias(in, 3, out, 5)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  if (int e = get_encode()) return e;
  const CpoLayout cl = cpo_layout(B, S, H, V);
  const BwdLayout lay = bwd_layout(T, H, V, cl.end);
  const FusedWs w = flce_ws_carve(ws, ws_bytes, T, V);
  const FlceBwdWs bw = bwd_carve(ws, lay);
  char* base = static_cast<char*>(ws);
  CpoArgs c{B, S, beta, alpha, reinterpret_cast<float*>(base + cl.off_lp), reinterpret_cast<float*>(base + cl.off_sig),
            reinterpret_cast<float*>(base + cl.off_mean), logps, reinterpret_cast<float*>(base + lay.end - kAlign)};
  FlceBwdMaps m;
  if (tmap_bf16(&m.x, x, T, H, kBM) || tmap_bf16(&m.w, W, V, H, kBoxBFwd) ||
      tmap_bf16_ld(&m.dz, bw.dz, T, V, bw.ld_dz, kBM) || tmap_bf16_mn(&m.w_mn, W, V, H, H, kBoxBGrad) ||
      tmap_bf16_mn(&m.dz_mn, bw.dz, T, V, bw.ld_dz, kBM) || tmap_bf16_mn(&m.x_mn, x, T, H, H, kBoxBGrad))
    return LMHO_ERR_CUDA;
  const FusedGeometry g = geometry(T, H, V, kBN_CE);
  const FusedLaunch L{sms, g_timeout_ns.load(), static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_flce_fwd_bwd(m, target, g, grad_scale, loss, dx, dW, w, bw, L, &c));
}

int lmho_probe_read(const void* data, int64_t segments, int64_t segment_bytes, uint32_t* out, void* stream) {
  if (!data || !out || segments <= 0 || segment_bytes <= 0 || segment_bytes % 16 != 0) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(data) || segments > (int64_t(1) << 31) - 2) return LMHO_ERR_INVALID_ARG;
  const Range in[1] = {rng(data, static_cast<size_t>(segments) * static_cast<size_t>(segment_bytes))};
  const Range out_r[1] = {rng(out, 4 * static_cast<size_t>(segments))};
  if (int a = check_alias(in, 1, out_r, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_probe_read(data, segments, segment_bytes, out, static_cast<cudaStream_t>(stream)));
}

int lmho_copy_h2d(void* dst, const void* src, int64_t bytes, void* stream) {
  if (bytes < 0) return LMHO_ERR_INVALID_ARG;
  if (bytes == 0) return LMHO_OK;
  if (!dst || !src || bytes % 16 != 0 || !aligned16(dst) || !aligned16(src)) return LMHO_ERR_INVALID_ARG;
  const Range in[1] = {rng(src, static_cast<size_t>(bytes))};
  const Range out_r[1] = {rng(dst, static_cast<size_t>(bytes))};
  if (int a = check_alias(in, 1, out_r, 1)) return a;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  // src: pinned host memory with a device mapping; dst: memory the GPU owns
  cudaPointerAttributes as{}, ad{};
  if (cudaPointerGetAttributes(&as, src) != cudaSuccess || cudaPointerGetAttributes(&ad, dst) != cudaSuccess) {
    (void)cudaGetLastError();
    return LMHO_ERR_INVALID_ARG;
  }
  if (as.type != cudaMemoryTypeHost || !as.devicePointer) return LMHO_ERR_INVALID_ARG;
  if (ad.type != cudaMemoryTypeDevice && ad.type != cudaMemoryTypeManaged) return LMHO_ERR_INVALID_ARG;
  if (!aligned16(as.devicePointer)) return LMHO_ERR_INVALID_ARG;
  const int blocks = sms / 2 > 0 ? sms / 2 : 1;
  return cuda_status(launch_copy_h2d(as.devicePointer, dst, bytes, blocks, static_cast<cudaStream_t>(stream)));
}

int lmho_ws_status(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kAlign || !aligned256(ws)) return LMHO_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LMHO_ERR_CUDA;
  Ctrl* c = ctrl_of(ws, ws_bytes);
  uint32_t st = 0;
  if (cudaMemcpy(&st, &c->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LMHO_ERR_CUDA;
  if (st != 0) {
    if (cudaMemset(&c->status, 0, 4) != cudaSuccess) return LMHO_ERR_CUDA;
    return static_cast<int>(st);
  }
  return LMHO_OK;
}

int lmho_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, void* stream) {
  if (!ws || ws_bytes < kAlign || !aligned256(ws)) return LMHO_ERR_INVALID_ARG;
  int sms = 0;
  if (int d = current_device(&sms)) return d;
  return cuda_status(launch_wait_selftest(ctrl_of(ws, ws_bytes), timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
