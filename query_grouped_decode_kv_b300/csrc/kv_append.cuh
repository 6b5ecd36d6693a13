// kv_append.cuh -- write this step's K/V rows into the cache (bit copy, 16 bytes per thread).
//
// Definition: "分组查询注意力（GQA）与多查询注意力（MQA）深度实战" (ybb.press) §八 stores the new
// token's K/V rows of the g KV heads at the current position; nanhubrain.csdn.net's MQA article
// §2.2 appends the new row along the sequence axis. Here the position is per sequence.
#pragma once

#include <stdint.h>

#include "status.cuh"

namespace mqa {

// One thread moves one 16-byte chunk of one (sequence, KV head) row of K and the matching chunk
// of V. Rows whose position is out of range are skipped and latch MQA_ERR_DEVICE_BOUNDS.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        uint4* __restrict__ k_cache,
                                                        uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ pos, int b,
                                                        int g, int chunks_per_row, int n_max) {
  const long long total = static_cast<long long>(b) * g * chunks_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long row = idx / chunks_per_row;  // = bi * g + j
    const int c = static_cast<int>(idx - row * chunks_per_row);
    const int bi = static_cast<int>(row / g);
    const int p = __ldg(pos + bi);
    if (p < 0 || p >= n_max) {
      if (c == 0 && row == static_cast<long long>(bi) * g) latch_status(kStatusDeviceBounds);
      continue;
    }
    const long long dst = (row * n_max + p) * chunks_per_row + c;
    k_cache[dst] = __ldg(k_new + idx);
    v_cache[dst] = __ldg(v_new + idx);
  }
}

}  // namespace mqa
