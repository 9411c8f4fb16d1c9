// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cstdint>

namespace slm {

// Bits of the device status word (int32) that kernels OR into *dev_status.
constexpr int32_t kDevBadSeqlens = 1;        // sequence boundary not non-decreasing / not ending at T
constexpr int32_t kDevBadParent = 2;         // parent index outside [0, W)
constexpr int32_t kDevPipelineTimeout = 4;   // a bounded wait inside a kernel ran out

}  // namespace slm
