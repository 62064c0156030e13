// Host -> device copy done by the SMs: each thread loads 16-byte words of the
// pinned host buffer through its device mapping and stores them to device
// memory.  Kept off the copy engines on purpose: on GB300 with its Grace host,
// copy-engine transfers from pinned memory were repeatedly slowed by bursts
// of host page faults that the SM loads do not cause once their mappings are
// in place; a small grid (half the SMs, 128 threads each) carries the host
// link's rate while leaving most of each SM to the kernels it runs beside.
#include "transfer.h"

namespace lmho {
namespace {

constexpr int kCopyThreads = 128;
constexpr int kCopyUnroll = 8;   // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads)
    copy_h2d_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // whole rounds: kCopyUnroll words per thread, the last at i + (kCopyUnroll - 1) stride < n
  for (; i + (kCopyUnroll - 1) * stride < n; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) __stcs(dst + i + k * stride, v[k]);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace

cudaError_t launch_copy_h2d(const void* src, void* dst, int64_t bytes, int blocks, cudaStream_t st) {
  copy_h2d_kernel<<<static_cast<unsigned>(blocks), kCopyThreads, 0, st>>>(static_cast<const uint4*>(src),
                                                                           static_cast<uint4*>(dst), bytes / 16);
  return cudaGetLastError();
}

}  // namespace lmho
