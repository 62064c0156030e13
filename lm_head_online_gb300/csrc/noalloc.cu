// ce_fwd_f32_noalloc: the flat fp32 cross-entropy for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or not at the moment they need
// the loss: callers that own a fixed device-memory budget (a serving process
// that reserved its pool up front, a plug-in loaded into someone else's
// allocator, which must not grow the device footprint behind that allocator's
// back), or bindings that have no device allocator to hand.  ce_fwd_f32 asks
// them for a workspace; this variant instead uses scratch memory owned by the
// library: one file-scope __device__ array, sized for at most
// kNoAllocMaxTokens tokens, that every GPU which loads the library keeps for
// the life of the process.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no library routine that
// allocates.  The row decomposition is ce_fwd_f32's (the same automatic rule,
// or the same process-wide override), so are the kernels; only the scratch
// pointers differ.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/lmho.h"
#include "lmho_internal.h"
#include "ptx.cuh"

namespace lmho {
namespace {

// Per-token losses of up to kNoAllocMaxTokens rows, then one 256-byte control
// block (status word; the ticket word is unused by this call).
constexpr int64_t kNoAllocMaxTokens = 65536;
constexpr size_t kNoAllocRowBytes = 4 * kNoAllocMaxTokens;
constexpr size_t kNoAllocScratchBytes = kNoAllocRowBytes + sizeof(Ctrl);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host code cannot use g_noalloc_scratch as an address (on the host it names a
// shadow variable, not device memory).  Its device address is looked up with
// cudaGetSymbolAddress, with the device current, and cached per device
// together with the id of the context it was looked up in: a new context on
// that device (after cudaDeviceReset, or a released primary context) reloads
// the module, so the address is looked up again instead of reusing a stale one.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_pfn_once;

void load_driver_queries() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Id of the calling thread's current context, or 0 if there is none.
unsigned long long current_ctx_id() {
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct Cached {
  void* ptr = nullptr;
  unsigned long long ctx = 0;
};
std::mutex g_mu;
Cached g_scratch[kMaxDevices];

int scratch_address(int dev, void** out) {
  std::call_once(g_pfn_once, load_driver_queries);
  if (!g_ctx_current || !g_ctx_id) return LMHO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Cached& c = g_scratch[dev];
  const unsigned long long now = current_ctx_id();
  if (!c.ptr || now == 0 || now != c.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LMHO_ERR_CUDA;
    const unsigned long long after = current_ctx_id();   // the lookup makes the device's context current
    if (after == 0) return LMHO_ERR_CUDA;
    c.ptr = p;
    c.ctx = after;
  }
  *out = c.ptr;
  return LMHO_OK;
}

}  // namespace
}  // namespace lmho

using namespace lmho;

extern "C" int ce_fwd_f32_noalloc(const float* logits, const int64_t* target, int64_t T, int64_t V, float* loss,
                                  void* stream) {
  if (!logits || !target || !loss) return LMHO_ERR_INVALID_ARG;
  if (T <= 0 || V <= 0 || T > kNoAllocMaxTokens) return LMHO_ERR_INVALID_ARG;
  const uintptr_t z0 = reinterpret_cast<uintptr_t>(logits), z1 = z0 + 4 * static_cast<uintptr_t>(T) * V;
  const uintptr_t t0 = reinterpret_cast<uintptr_t>(target), t1 = t0 + 8 * static_cast<uintptr_t>(T);
  const uintptr_t l0 = reinterpret_cast<uintptr_t>(loss), l1 = l0 + 4;
  if ((l0 < z1 && z0 < l1) || (l0 < t1 && t0 < l1)) return LMHO_ERR_ALIAS;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LMHO_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LMHO_ERR_CUDA;
  if (major != 10 || minor != 3) return LMHO_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (int e = scratch_address(dev, &scratch)) return e;
  float* row_loss = static_cast<float*>(scratch);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(static_cast<char*>(scratch) + kNoAllocRowBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The scratch keeps whatever the previous call left: clear the control
  // block (its status word must start at zero) first.
  if (cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st) != cudaSuccess) return LMHO_ERR_CUDA;
  return launch_ce_f32(logits, target, T, V, loss, row_loss, ctrl, choose_ce(logits, T, V, 4, sms), st) ==
                 cudaSuccess
             ? LMHO_OK
             : LMHO_ERR_CUDA;
}
