// kv_append.cuh -- write this step's K/V rows into the cache (bit copy, 16 bytes per thread).
//
// Definition: "分组查询注意力（GQA）与多查询注意力（MQA）深度实战" (ybb.press) §八 stores the new
// token's K/V rows of the g KV heads at the current position; nanhubrain.csdn.net's MQA article
// §2.2 appends the new row along the sequence axis. Here the position is per sequence.
#pragma once

#include <stdint.h>

#include "decode_attention.cuh"
#include "status.cuh"

namespace mqa {

// One thread moves one 16-byte chunk of one (sequence, token, KV head) row of K and the matching
// chunk of V: token t of sequence bi goes to row pos[bi] + t. A sequence whose rows
// pos .. pos + T - 1 are not all in range is skipped and latches MQA_ERR_DEVICE_BOUNDS.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        uint4* __restrict__ k_cache,
                                                        uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ pos, int b,
                                                        int T, int g, int chunks_per_row,
                                                        int n_max) {
  const long long total = static_cast<long long>(b) * T * g * chunks_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long src_row = idx / chunks_per_row;  // = (bi * T + t) * g + j
    const int c = static_cast<int>(idx - src_row * chunks_per_row);
    const long long bt = src_row / g;
    const int j = static_cast<int>(src_row - bt * g);
    const int bi = static_cast<int>(bt / T);
    const int t = static_cast<int>(bt - static_cast<long long>(bi) * T);
    const int p = __ldg(pos + bi);
    if (p < 0 || static_cast<long long>(p) + T > n_max) {
      if (c == 0 && t == 0 && j == 0) latch_status(kStatusDeviceBounds);
      continue;
    }
    const long long dst =
        ((static_cast<long long>(bi) * g + j) * n_max + p + t) * chunks_per_row + c;
    k_cache[dst] = __ldg(k_new + idx);
    v_cache[dst] = __ldg(v_new + idx);
  }
}

// The same append into paged caches: pools [num_pages][g][page_size][chunks] of 16-byte chunks,
// row p of sequence bi living at row p % page_size of page page_table[bi][p / page_size]
// (the nanhubrain.csdn.net MQA article §3.3: vLLM keeps the cache in fixed pages, 16 tokens each
// by default; "GQA与MQA深度实战" (ybb.press) §十 item 12 pairs ragged batches with such paging).
// A position outside [0, max_pages * page_size) or a page index outside [0, num_pages) skips that
// sequence and latches MQA_ERR_DEVICE_BOUNDS.
__global__ void __launch_bounds__(256) kv_append_paged_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ page_table, int b, int g, int chunks_per_row, int page_size,
    int max_pages, int num_pages) {
  const long long total = static_cast<long long>(b) * g * chunks_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long n_max = static_cast<long long>(max_pages) * page_size;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long row = idx / chunks_per_row;  // = bi * g + j
    const int c = static_cast<int>(idx - row * chunks_per_row);
    const int bi = static_cast<int>(row / g);
    const int j = static_cast<int>(row - static_cast<long long>(bi) * g);
    const int p = __ldg(pos + bi);
    const bool first = c == 0 && j == 0;
    if (p < 0 || p >= n_max) {
      if (first) latch_status(kStatusDeviceBounds);
      continue;
    }
    const int page = __ldg(page_table + static_cast<size_t>(bi) * max_pages + p / page_size);
    if (page < 0 || page >= num_pages) {
      if (first) latch_status(kStatusDeviceBounds);
      continue;
    }
    const long long dst =
        ((static_cast<long long>(page) * g + j) * page_size + p % page_size) * chunks_per_row + c;
    k_pool[dst] = __ldg(k_new + idx);
    v_pool[dst] = __ldg(v_new + idx);
  }
}

// The append of T rows per sequence through the page table, into bf16 pools (EB = 2: a bit
// copy) or fp8 E4M3 pools (EB = 1: the codes e4m3(x / scale), the division rounded once in fp32).
// One thread writes one 16-byte chunk of one (sequence, token, KV head) row: token t of sequence
// bi goes to row p = pos[bi] + t, found at row p % page_size of page page_table[bi][p /
// page_size]. A sequence whose rows pos .. pos + T - 1 are not all in [0, max_pages * page_size)
// is skipped; a row whose page index is out of range is skipped alone; both latch
// MQA_ERR_DEVICE_BOUNDS. (The fused step writes its new rows with the same rules.)
template <int EB>
__global__ void __launch_bounds__(256) kv_append_paged_rows_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int32_t* __restrict__ pos,
    const int32_t* __restrict__ page_table, int b, int T, int g, int d_h, int page_size,
    int max_pages, int num_pages, float k_scale, float v_scale) {
  const int ch = d_h * EB / 16;  // 16-byte chunks per pool row
  const int cs = d_h / 8;        // 16-byte chunks per source row (bf16)
  const long long total = static_cast<long long>(b) * T * g * ch;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long n_max = static_cast<long long>(max_pages) * page_size;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long src_row = idx / ch;  // = (bi * T + t) * g + j
    const int c = static_cast<int>(idx - src_row * ch);
    const long long bt = src_row / g;
    const int j = static_cast<int>(src_row - bt * g);
    const int bi = static_cast<int>(bt / T);
    const int t = static_cast<int>(bt - static_cast<long long>(bi) * T);
    const int p0 = __ldg(pos + bi);
    if (p0 < 0 || static_cast<long long>(p0) + T > n_max) {
      if (c == 0 && t == 0 && j == 0) latch_status(kStatusDeviceBounds);
      continue;
    }
    const int p = p0 + t;
    const int page = __ldg(page_table + static_cast<size_t>(bi) * max_pages + p / page_size);
    if (page < 0 || page >= num_pages) {
      if (c == 0 && j == 0) latch_status(kStatusDeviceBounds);
      continue;
    }
    const long long dst =
        ((static_cast<long long>(page) * g + j) * page_size + p % page_size) * ch + c;
    k_pool[dst] = new_row_chunk<EB>(k_new + src_row * cs, c, k_scale);
    v_pool[dst] = new_row_chunk<EB>(v_new + src_row * cs, c, v_scale);
  }
}

// The append into fp8 E4M3 caches [b][g][n_max][D] (one byte per element): one thread writes one
// 16-byte chunk of codes, e4m3(x / scale) for 16 consecutive bf16 values x of the new row (the
// division rounded once in fp32, nearest-even rounding to E4M3 saturating at +-448). Positions
// out of range skip the sequence and latch MQA_ERR_DEVICE_BOUNDS.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int32_t* __restrict__ pos, int b, int g, int d_h,
    int n_max, float k_scale, float v_scale) {
  const int ch = d_h / 16;   // output chunks per row
  const int cs = d_h / 8;    // source chunks per row
  const long long total = static_cast<long long>(b) * g * ch;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long row = idx / ch;  // = bi * g + j
    const int c = static_cast<int>(idx - row * ch);
    const int bi = static_cast<int>(row / g);
    const int p = __ldg(pos + bi);
    if (p < 0 || p >= n_max) {
      if (c == 0 && row == static_cast<long long>(bi) * g) latch_status(kStatusDeviceBounds);
      continue;
    }
    const long long dst = (row * n_max + p) * ch + c;
    k_cache[dst] = new_row_chunk<1>(k_new + row * cs, c, k_scale);
    v_cache[dst] = new_row_chunk<1>(v_new + row * cs, c, v_scale);
  }
}

}  // namespace mqa
