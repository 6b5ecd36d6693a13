// status.cuh -- the per-device status word that kernels latch errors into.
#pragma once

namespace mqa {

// Values mirror mqa_status in include/mqa.h.
constexpr int kStatusOk = 0;
constexpr int kStatusDeviceBounds = 4;
constexpr int kStatusTimeout = 5;

// One word per device (this module's copy of the variable lives on every device that loads the
// library). The first error wins; the host reads and clears it in mqa_get_device_status().
__device__ int g_device_status = 0;

__device__ __forceinline__ void latch_status(int code) { atomicCAS(&g_device_status, 0, code); }

}  // namespace mqa
