// Host -> device transfer by the SMs (lmho_copy_h2d).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace lmho {

// Copies `bytes` (a multiple of 16) from `src`, a device-side address of
// pinned host memory, to device memory `dst` (both 16-byte aligned) with one
// grid-stride kernel of `blocks` blocks on `st`.
cudaError_t launch_copy_h2d(const void* src, void* dst, int64_t bytes, int blocks, cudaStream_t st);

}  // namespace lmho
