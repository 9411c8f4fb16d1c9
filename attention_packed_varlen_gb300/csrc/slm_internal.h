// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace slm {

// Launch configuration for a programmatic dependent of the kernel before it
// on the stream (griddepcontrol.wait in the kernel orders its memory accesses
// after that kernel; its setup may overlap that kernel's tail).
inline cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, dim3 grid, dim3 block, cudaStream_t stream,
                                     size_t smem = 0) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Bits of the device status word (int32) that kernels OR into *dev_status.
constexpr int32_t kDevBadSeqlens = 1;        // sequence boundary not non-decreasing / not ending at T
constexpr int32_t kDevBadParent = 2;         // parent index outside [0, W)
constexpr int32_t kDevPipelineTimeout = 4;   // a bounded wait inside a kernel ran out
constexpr int32_t kDevBounds = 8;            // debug-bounds builds: an index outside its buffer

#if defined(__CUDACC__)
// Builds with -DSLM_DEBUG_BOUNDS check the indices the kernels compute
// against the buffers they address: a failed check ORs kDevBounds into the
// status word and the caller skips the access (it never traps).  Other builds
// compile the checks away.
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* status) {
#ifdef SLM_DEBUG_BOUNDS
  if (!ok && status) atomicOr(status, kDevBounds);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}
#endif

}  // namespace slm
