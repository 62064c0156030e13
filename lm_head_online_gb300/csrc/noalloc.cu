// ce_fwd_f32_noalloc: the flat fp32 cross-entropy for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or not at the moment they need
// the loss: code running while a CUDA graph is being captured, callers that
// own a fixed device-memory budget (a serving process that reserved its pool
// up front, a plug-in loaded into someone else's allocator), or bindings that
// have no device allocator to hand.  ce_fwd_f32 asks them for a workspace;
// this variant instead uses scratch memory owned by the library: one
// file-scope __device__ array, sized for at most kNoAllocMaxTokens tokens, that
// every GPU which loads the library keeps for the life of the process.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no library routine that
// allocates.  The kernels are the ones ce_fwd_f32 launches; only the scratch
// pointers differ.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/lmho.h"
#include "lmho_internal.h"
#include "ptx.cuh"

namespace lmho {
namespace {

// Per-token losses of up to kNoAllocMaxTokens rows, then one 256-byte control
// block (ticket of the last-block mean, status word).
constexpr int64_t kNoAllocMaxTokens = 65536;
constexpr size_t kNoAllocRowBytes = 4 * kNoAllocMaxTokens;
constexpr size_t kNoAllocScratchBytes = kNoAllocRowBytes + sizeof(Ctrl);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host code cannot use g_noalloc_scratch as an address (on the host it names a
// shadow variable, not device memory); its device address is looked up once
// per device, with that device current, and cached here.
std::mutex g_mu;
void* g_scratch_dev[64] = {};

int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LMHO_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return LMHO_OK;
}

CeConfig noalloc_config(int64_t V) {
  // same rule as ce_fwd_f32's automatic choice for these row counts
  return (V * 4 <= 16 * 1024) ? CeConfig{kCeWarp, 256, 1} : CeConfig{kCeCta, 256, 1};
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

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LMHO_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return LMHO_ERR_CUDA;
  if (major != 10 || minor != 3) return LMHO_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (int e = scratch_address(dev, &scratch)) return e;
  float* row_loss = static_cast<float*>(scratch);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(static_cast<char*>(scratch) + kNoAllocRowBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The scratch keeps whatever the previous call left: the ticket of the
  // last-block mean must start at zero, so clear the control block first.
  if (cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st) != cudaSuccess) return LMHO_ERR_CUDA;
  return launch_ce_f32(logits, target, T, V, loss, row_loss, ctrl, noalloc_config(V), st) == cudaSuccess
             ? LMHO_OK
             : LMHO_ERR_CUDA;
}
