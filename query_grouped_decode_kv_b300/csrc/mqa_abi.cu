// mqa_abi.cu -- the extern "C" entry points declared in include/mqa.h: host-side argument
// checks, the per-(device, stream) workspace, TMA descriptors, and kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/mqa.h"
#include "decode_attention.cuh"
#include "decode_attention_tc.cuh"
#include "kv_append.cuh"
#include "prefill_attention_tc.cuh"
#include "status.cuh"

namespace {

using mqa::DecodeParams;

std::atomic<uint64_t> g_launches{0};
// Bumped each time mqa_get_device_status reports MQA_ERR_TIMEOUT: a kernel that gave up may have
// left arrival counters non-zero, so every scratch area clears them once more before its next use.
std::atomic<uint64_t> g_timeout_epoch{0};
std::atomic<int> g_force_ctas{0};
std::atomic<int> g_force_path{0};

constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s per wait
// The in-kernel wait limit in force (testing hook: mqa_debug_set_wait_limit_ns); the waits for a
// CTA's own copies and MMAs in flight at exit always keep kWaitLimitNs.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int> g_debug_stall{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
// ------------------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Cache [b][g][n_max][d_h] seen as a 3-D tensor (d_h, n_max, b*g) of bf16 (eb = 2) or of
// one-byte fp8 codes (eb = 1); box = 128 bytes of columns x kTileKeys rows, 128-byte swizzle.
// Rows past n_max read as zeros.
bool make_cache_map(CUtensorMap* map, const void* base, int bg, int n_max, int d_h, int eb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d_h), static_cast<cuuint64_t>(n_max),
                              static_cast<cuuint64_t>(bg)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_h) * eb,
                                 static_cast<cuuint64_t>(n_max) * d_h * eb};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(mqa::kSwizzleRowBytes / eb), mqa::kTileKeys,
                             1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A page pool [num_pages][g][page_size][d_h] bf16 seen as (d_h, page_size, num_pages * g); box =
// 64 columns x min(page_size, kTileKeys) rows, 128-byte swizzle. Coordinates past the pool read
// as zeros.
bool make_pool_map(CUtensorMap* map, const void* base, long long pages_g, int page_size,
                   int d_h, int eb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d_h), static_cast<cuuint64_t>(page_size),
                              static_cast<cuuint64_t>(pages_g)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_h) * eb,
                                 static_cast<cuuint64_t>(page_size) * d_h * eb};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(mqa::kSwizzleRowBytes / eb),
                             static_cast<cuuint32_t>(page_size < mqa::kTileKeys
                                                         ? page_size : mqa::kTileKeys), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Paged caches: the page table and the pool's geometry (all zero for contiguous caches).
struct PagedCache {
  const int32_t* table = nullptr;
  int page_size = 0, max_pages = 0, num_pages = 0;
};

// Host checks shared by the paged entry points. Page sizes: powers of two from 8 rows. With 8, 16
// or 32 rows a tile of 64 rows spans several pages, one bulk copy each (a box of 8 or more rows
// keeps every copy on a 1 KB boundary of the stage, where the 128-byte swizzle repeats); from 64
// rows every tile lies inside one page. Sets *n_max to the rows a sequence can address.
int check_paged(const PagedCache& pg, int g, int d_h, int* n_max) {
  if (!pg.table || (reinterpret_cast<uintptr_t>(pg.table) & 3u)) return MQA_ERR_INVALID_ARG;
  if (pg.page_size <= 0 || pg.max_pages <= 0 || pg.num_pages <= 0) return MQA_ERR_INVALID_ARG;
  if (pg.page_size < 8 || (pg.page_size & (pg.page_size - 1)) != 0) return MQA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(pg.max_pages) * pg.page_size;
  if (rows > 0x7fffffffll) return MQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(pg.num_pages) * g > 0x7fffffffll - 1) return MQA_ERR_UNSUPPORTED;
  if (static_cast<double>(pg.num_pages) * g * pg.page_size * d_h > 9.0e18)
    return MQA_ERR_UNSUPPORTED;
  *n_max = static_cast<int>(rows);
  return MQA_OK;
}

// ------------------------------------------------------------------------------------------------
// Workspace, one per (device, stream), growing on demand. Two separate buffers: the split partial
// states (written before they are read in every call), and one arrival counter per segment. The
// counters must read zero when a call starts: a new counter buffer is zeroed, every call that
// finishes leaves its counters at zero, and nothing else ever writes there.
//
// Each buffer is two halves, and consecutive launches on the stream take alternate halves. A
// launch that overlaps the one ahead of it (early writes) then never shares scratch with it; the
// launch two back, which used the same half, has finished before it starts (its launch-order
// warp sees to that).
// ------------------------------------------------------------------------------------------------
struct DeviceBuffer {
  void* ptr = nullptr;
  size_t bytes = 0;
};
struct Workspace {
  DeviceBuffer partials, counters;
  uint64_t clean_epoch = 0;  // g_timeout_epoch when its counters were last known to be zero
  uint32_t launches = 0;     // launches on this stream so far: the half the next one takes
};
std::mutex g_ws_mutex;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

// Grow `buf` to at least `bytes` (with 25% headroom); zero the new buffer when `zero`.
int grow_buffer(DeviceBuffer& buf, size_t bytes, cudaStream_t stream, bool zero) {
  if (buf.bytes >= bytes) return MQA_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MQA_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return MQA_ERR_UNSUPPORTED;  // cannot grow in capture
  if (buf.ptr) {
    // the old buffer may still be used by earlier work on this stream
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MQA_ERR_CUDA;
    cudaFree(buf.ptr);
    buf.ptr = nullptr;
    buf.bytes = 0;
  }
  const size_t grow = bytes + bytes / 4;
  if (cudaMalloc(&buf.ptr, grow) != cudaSuccess) {
    buf.ptr = nullptr;
    return MQA_ERR_CUDA;
  }
  if (zero && cudaMemsetAsync(buf.ptr, 0, grow, stream) != cudaSuccess) return MQA_ERR_CUDA;
  buf.bytes = grow;
  return MQA_OK;
}

// The scratch a launch uses: the partial states, the arrival counters, whether the whole
// counter region (`counter_region`, `counter_region_bytes`: all the counters any call may use
// there, both halves of a workspace) must be zeroed first, and whether the scratch is not shared
// with the launch ahead on the stream (a workspace half), so that the launch may write early.
struct Scratch {
  void* partials = nullptr;
  unsigned int* counters = nullptr;
  void* counter_region = nullptr;
  size_t counter_region_bytes = 0;
  bool clear = false;
  bool alternating = false;
};

int get_workspace(int dev, cudaStream_t stream, size_t partial_bytes, size_t counter_bytes,
                  Scratch* out) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace& ws = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
  // two halves of each buffer, every half at least this call's need, 256-byte aligned
  const size_t half_p = (partial_bytes + 255) & ~size_t{255};
  const size_t half_c = (counter_bytes + 255) & ~size_t{255};
  if (int st = grow_buffer(ws.partials, 2 * half_p, stream, false)) return st;
  const uint64_t epoch = g_timeout_epoch.load();
  if (ws.counters.bytes < 2 * half_c) {
    if (int st = grow_buffer(ws.counters, 2 * half_c, stream, true)) return st;
    ws.clean_epoch = epoch;
  }
  // After a timeout any counter of the region may be dirty, not only the ones this call uses, so
  // the clear (and with it the clean mark) covers the whole region.
  out->clear = ws.clean_epoch != epoch;
  ws.clean_epoch = epoch;
  const uint32_t half = ws.launches++ & 1u;
  const size_t stride_p = (ws.partials.bytes / 2) & ~size_t{255};
  const size_t stride_c = (ws.counters.bytes / 2) & ~size_t{255};
  out->partials = static_cast<char*>(ws.partials.ptr) + half * stride_p;
  out->counters = reinterpret_cast<unsigned int*>(static_cast<char*>(ws.counters.ptr) +
                                                  half * stride_c);
  out->counter_region = ws.counters.ptr;
  out->counter_region_bytes = ws.counters.bytes;
  out->alternating = true;
  return MQA_OK;
}

// Streams whose decode-attention launches may overlap the kernel ahead of them
// (mqa_set_launch_overlap), keyed by (device, stream).
std::mutex g_overlap_mutex;
std::map<std::pair<int, uintptr_t>, bool> g_overlap;

bool overlap_on(int dev, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_overlap_mutex);
  auto it = g_overlap.find({dev, reinterpret_cast<uintptr_t>(stream)});
  return it != g_overlap.end() && it->second;
}

// Overlapped launches whose K and V caches together hold at most this many bytes (b*g*n_max rows
// of d_h elements, both caches) write early; larger ones wait before their first write. Measured
// on B300 with launches back to back, early writes against waiting: 18.0 us against 20.4 us per
// launch at b=8, h=32, g=8, contexts 512-4096 (134 MB of caches); 51.0 against 53.0 us at b=64,
// h=32, g=1, context 8192 (268 MB); 74.1-74.5 against 75.2 us over fp8 codes at b=8, h=64, g=8,
// contexts 1024-32768 (537 MB); the same shape over bf16 (1.07 GB) 98.8-102.0 against 98.4 us
// per layer across 80 layers.
constexpr double kEarlyWritesMaxCacheBytes = 768.0 * 1024 * 1024;

struct DeviceInfo {
  int sms = 0;
};
std::mutex g_dev_mutex;
std::map<int, DeviceInfo> g_dev;

int device_info(int dev, DeviceInfo* info) {
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MQA_ERR_CUDA;
    it = g_dev.emplace(dev, d).first;
  }
  *info = it->second;
  return MQA_OK;
}

// ------------------------------------------------------------------------------------------------
// Kernel selection
// ------------------------------------------------------------------------------------------------
using AttnKernel = void (*)(const CUtensorMap, const CUtensorMap, const DecodeParams);

// The inner-product paths (mqa_debug_override's `path`): CUDA cores, mma.sync tensor cores, and
// tcgen05 tensor cores with tensor-memory accumulators.
enum Path { kPathAuto = 0, kPathCudaCores = 1, kPathMmaSync = 2, kPathTcgen05 = 3 };

// Automatic choice, by measurement on B300. With one or two heads per K/V row (MHA-like
// grouping) the heads are no contraction and CUDA cores stream the cache at the HBM rate. From
// three heads on, the CUDA cores' fp32 FMAs (2 G d_h per key) fall behind HBM (at 32K rows:
// 1.01x the copy bandwidth at G = 3, 0.87x at G = 4, 0.59x at G = 7, against 1.10x on mma.sync at
// every G), so the group's heads go to the tensor cores (mma.sync m16n8k16: up to 8 heads as the
// N columns of transposed products, beyond that as M rows padded to 16; the tcgen05 kernel,
// 128-row MMA tiles with accumulators in tensor memory, is not faster on any measured decode
// shape). Forcing either path at any G up to 7 is supported and tested.
constexpr int kCudaCoreMaxGroup = 2;
Path auto_path(int G) { return G <= kCudaCoreMaxGroup ? kPathCudaCores : kPathMmaSync; }


// A kernel instance with the launch facts the host needs.
struct AttnKernelChoice {
  AttnKernel fn = nullptr;
  int threads = 0;
  size_t smem = 0;
  bool wide = false;  // eight consumer warps with a setmaxnreg split: check the register count
  bool pdl = false;   // writes global memory only after griddepcontrol.wait (may overlap)
};

template <class Consumer, int D, int EB, bool TC, int WM>
AttnKernelChoice choice(int b) {
  AttnKernelChoice c;
  c.fn = mqa::decode_attention_kernel<D, EB, Consumer, TC, WM>;
  c.threads = mqa::threads_of(Consumer::kWarps);
  c.smem = mqa::smem_bytes<D, EB, Consumer::kRingBytes>(Consumer::kWarps, Consumer::kCombRows);
  c.wide = Consumer::kWarps == 8;
  c.pdl = true;
  return c;
}

// Eight consumer warps (two per SM sub-partition) hide the latency of the per-tile dependency
// chains where one warp per sub-partition leaves most issue slots idle: the CUDA-core path, and
// mma.sync above 16 heads, where each warp's MMA chains and softmax would otherwise serialise.
// Up to 16 heads mma.sync keeps four warps (16 keys per warp is its smallest P V k-step).
template <int D>
AttnKernelChoice pick_kernel(Path path, int G, int b, int T) {
  using mqa::MmaConsumer;
  if (path == kPathTcgen05) {
    // the group's heads padded to 16, 32 or 64 rows of the 128-row MMA tile
    AttnKernelChoice c;
    c.fn = G <= 16 ? mqa::decode_attention_tc_kernel<D, 16>
                   : (G <= 32 ? mqa::decode_attention_tc_kernel<D, 32>
                              : mqa::decode_attention_tc_kernel<D, 64>);
    c.threads = mqa::kTcThreads;
    c.smem = mqa::tc_smem_bytes(D);
    return c;
  }
  if (path == kPathMmaSync && T > 1) {
    // rows = T x heads, each masked by its token's causal limit
    if (G <= 16) return choice<MmaConsumer<D, 1, 4, true>, D, 2, true, 1>(b);
    if (G <= 32) return choice<MmaConsumer<D, 2, 8, true>, D, 2, true, 2>(b);
    return choice<MmaConsumer<D, 4, 8, true>, D, 2, true, 4>(b);
  }
  if (path == kPathMmaSync) {
    // up to 8 heads, one token: the products transposed (heads on the MMA's 8 columns, no
    // padding rows). Measured on B300 against the head-row consumer, launches back to back:
    // gqa_8b 17.15 against 18.15 us, one 70B-class layer 99.9 against 100.9 us, the 80-layer
    // step in a graph 7,805 against 7,830 us.
    if (G <= 8) return choice<mqa::MmaConsumerT<D, 4>, D, 2, true, 1>(b);
    if (G <= 16) return choice<MmaConsumer<D, 1, 4>, D, 2, true, 1>(b);
    if (G <= 32) return choice<MmaConsumer<D, 2, 8>, D, 2, true, 2>(b);
    return choice<MmaConsumer<D, 4, 8>, D, 2, true, 4>(b);
  }
  switch (G) {
    case 1: return choice<mqa::CcConsumer2<D, 1>, D, 2, false, 1>(b);
    case 2: return choice<mqa::CcConsumer2<D, 2>, D, 2, false, 1>(b);
    case 3: return choice<mqa::CcConsumer2<D, 3>, D, 2, false, 1>(b);
    case 4: return choice<mqa::CcConsumer2<D, 4>, D, 2, false, 1>(b);
    case 5: return choice<mqa::CcConsumer2<D, 5>, D, 2, false, 1>(b);
    case 6: return choice<mqa::CcConsumer2<D, 6>, D, 2, false, 1>(b);
    case 7: return choice<mqa::CcConsumer2<D, 7>, D, 2, false, 1>(b);
    default: return {};
  }
}

// fp8 E4M3 caches (d_h = 128): the same paths with fp16 tensor-core MMAs or CUDA cores over the
// widened codes. The tcgen05 kernel does not read fp8 caches.
AttnKernelChoice pick_kernel_fp8(Path path, int G, int b) {
  using mqa::CcConsumer;
  using mqa::MmaConsumerF8;
  using mqa::MmaConsumerF8T;
  constexpr int D = 128;
  if (path == kPathTcgen05) return {};
  if (path == kPathMmaSync) {
    // several tile groups: an fp8 tile's HBM time is half a bf16 tile's while a warp's per-tile
    // chain is not shorter, so groups of warps take turns on the tiles. Up to 8 heads the
    // products run transposed (heads on the MMA's 8 columns, no padding rows). Measured on B300
    // (32K rows, launches back to back, fraction of the copy bandwidth on fp8 bytes): at G = 1-8
    // the transposed form reaches 0.90-0.91 with four groups of two warps (0.90-0.91 with eight
    // single warps, 0.82-0.83 with two groups of four) against 0.78-0.79 for the head-row form;
    // up to 16 heads four groups of two warps of the head-row form reach 0.77-0.79 against
    // 0.71-0.73 for two groups of four; at 32 heads two groups of four edge out one of eight
    // (0.456 against 0.449).
    if (G <= 8) return choice<MmaConsumerF8T<D, 8, 4>, D, 1, true, 1>(b);
    if (G <= 16) return choice<MmaConsumerF8<D, 1, 8, 4>, D, 1, true, 1>(b);
    if (G <= 32) return choice<MmaConsumerF8<D, 2, 8, 2>, D, 1, true, 2>(b);
    return choice<MmaConsumerF8<D, 4, 8>, D, 1, true, 4>(b);
  }
  switch (G) {
    case 1: return choice<CcConsumer<D, 1, 8, 1>, D, 1, false, 1>(b);
    case 2: return choice<CcConsumer<D, 2, 8, 1>, D, 1, false, 1>(b);
    case 3: return choice<CcConsumer<D, 3, 8, 1>, D, 1, false, 1>(b);
    case 4: return choice<CcConsumer<D, 4, 8, 1>, D, 1, false, 1>(b);
    case 5: return choice<CcConsumer<D, 5, 8, 1>, D, 1, false, 1>(b);
    case 6: return choice<CcConsumer<D, 6, 8, 1>, D, 1, false, 1>(b);
    case 7: return choice<CcConsumer<D, 7, 8, 1>, D, 1, false, 1>(b);
    default: return {};
  }
}

std::mutex g_attr_mutex;
std::map<std::pair<int, const void*>, size_t> g_smem_set;  // (device, kernel) -> bytes allowed

// Allow the kernel `bytes` of dynamic shared memory, and on first use check its register count:
// the eight-consumer-warp kernels move registers between warpgroups (setmaxnreg), which only
// completes if the launch allocated what the split assumes. A kernel built otherwise is refused
// rather than launched.
int prepare_kernel(int dev, const AttnKernelChoice& kc, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  const void* fn = reinterpret_cast<const void*>(kc.fn);
  auto it = g_smem_set.find({dev, fn});
  if (it == g_smem_set.end()) {
    if (kc.wide) {
      cudaFuncAttributes attr{};
      if (cudaFuncGetAttributes(&attr, fn) != cudaSuccess) return MQA_ERR_CUDA;
      if (attr.numRegs != mqa::kLaunchRegsWide) return MQA_ERR_UNSUPPORTED;
    }
    it = g_smem_set.emplace(std::make_pair(dev, fn), size_t{0}).first;
  }
  if (it->second >= bytes) return MQA_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return MQA_ERR_CUDA;
  it->second = bytes;
  return MQA_OK;
}

int launch_error() { return cudaGetLastError() == cudaSuccess ? MQA_OK : MQA_ERR_CUDA; }

// ------------------------------------------------------------------------------------------------
// Decode attention: host checks and launch plan, then the launch itself with a given scratch area
// (the split partial states: part_o [slots][G][d_h] fp32 followed by part_ml [slots][G] float2).
// ------------------------------------------------------------------------------------------------
struct DecodePlan {
  const mqa_bf16 *q, *k_cache, *v_cache;
  const int32_t* seq_lens;
  mqa_bf16* out;
  // fused append (mqa_decode_step only; null otherwise)
  const mqa_bf16 *k_new = nullptr, *v_new = nullptr;
  const int32_t* pos = nullptr;
  PagedCache paged;  // table null: contiguous caches
  int eb = 2;        // cache bytes per element: 2 bf16, 1 fp8 E4M3 codes
  int T = 1, Gh = 0; // new tokens per sequence; query heads per KV head (G = T * Gh rows)
  float k_scale = 1.f, v_scale = 1.f;  // fp8 caches: value = code * scale
  int b, h, g, d_h, n_max, G;
  float scale;
  Path path;
  bool prefill = false;  // several tokens with more than 64 rows per KV head: the prefill kernel
  bool path_forced = false;  // mqa_debug_override chose the inner-product path
  cudaStream_t stream;
  int dev;
  long long bg, ctas;
  // scratch, needed only with more than one CTA: partial states (part_o then part_ml) and one
  // arrival counter per segment, kept in a region of its own
  size_t part_o_bytes, partial_bytes, counter_bytes;
};

int plan_decode(const mqa_bf16* q, const mqa_bf16* k_cache, const mqa_bf16* v_cache,
                const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h, int n_max,
                float scale, void* stream, DecodePlan* plan, int T = 1) {
  // ---- host checks (no CUDA call before this block is done) ----
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || h <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return MQA_ERR_INVALID_ARG;
  if (h % g != 0) return MQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return MQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return MQA_ERR_INVALID_ARG;
  if (T <= 0) return MQA_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  const int Gh = h / g;
  const int force_path = g_force_path.load();
  // rows of a segment: the group's heads for each of the T tokens. Up to 64 of them run on the
  // decode kernels; several tokens with more rows (or with the tcgen05 path forced) run on the
  // prefill kernel, 128 rows per tensor-core tile.
  const long long rows = static_cast<long long>(T) * Gh;
  const bool prefill = T > 1 && (rows > mqa::kMaxGroup || force_path == kPathTcgen05);
  if ((!prefill && rows > mqa::kMaxGroup) || b > mqa::kMaxBatch) return MQA_ERR_UNSUPPORTED;
  if (prefill && (rows > mqa::kMaxPrefillRows ||
                  (force_path != kPathAuto && force_path != kPathTcgen05)))
    return MQA_ERR_UNSUPPORTED;
  const int G = static_cast<int>(rows);
  const long long bg = static_cast<long long>(b) * g;
  const long long tiles_per_seg =
      (static_cast<long long>(n_max) + mqa::kTileKeys - 1) / mqa::kTileKeys;
  if (bg > (1ll << 24) || static_cast<long long>(b) * tiles_per_seg >= (1ll << 31) ||
      static_cast<double>(bg) * n_max * d_h > 9.0e18)
    return MQA_ERR_UNSUPPORTED;
  // several tokens on the decode kernels: only the mma.sync consumer masks rows by token
  const Path path = prefill ? kPathTcgen05
                            : (force_path == kPathAuto ? (T > 1 ? kPathMmaSync : auto_path(G))
                                                       : static_cast<Path>(force_path));
  if (path == kPathCudaCores && G > 7) return MQA_ERR_UNSUPPORTED;
  if (T > 1 && !prefill && path != kPathMmaSync) return MQA_ERR_UNSUPPORTED;

  // ---- device facts ----
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MQA_ERR_CUDA;
  DeviceInfo info;
  if (int st = device_info(dev, &info)) return st;

  // CTAs: one per SM, but no more than a quarter of the (upper bound on the) tile count, so that
  // tiny problems are not scattered into many partial states. The prefill kernel: two per SM, at
  // most one per unit (128 rows of one sequence and KV head); it keeps no partial states.
  const long long w_max = bg * tiles_per_seg;
  const long long units = bg * ((rows + mqa::kPfRows - 1) / mqa::kPfRows);
  if (prefill && units >= (1ll << 31)) return MQA_ERR_UNSUPPORTED;
  long long ctas = prefill ? units : (w_max + 3) / 4;
  const long long max_ctas = prefill ? static_cast<long long>(mqa::kPfCtasPerSm) * info.sms
                                     : info.sms;
  if (ctas > max_ctas) ctas = max_ctas;
  if (ctas < 1) ctas = 1;
  if (const int f = g_force_ctas.load()) ctas = f;

  const long long slots = ctas + bg;
  DecodePlan& p = *plan;
  p.q = q; p.k_cache = k_cache; p.v_cache = v_cache; p.seq_lens = seq_lens; p.out = out;
  p.b = b; p.h = h; p.g = g; p.d_h = d_h; p.n_max = n_max; p.G = G;
  p.T = T; p.Gh = Gh;
  p.scale = scale;
  p.path = path;
  p.stream = static_cast<cudaStream_t>(stream);
  p.dev = dev;
  p.bg = bg;
  p.ctas = ctas;
  p.prefill = prefill;
  p.path_forced = force_path != kPathAuto;
  const bool split = ctas > 1 && !prefill;
  p.part_o_bytes = split ? static_cast<size_t>(slots) * G * d_h * sizeof(float) : 0;
  p.partial_bytes = split ? p.part_o_bytes + static_cast<size_t>(slots) * G * sizeof(float2) : 0;
  p.counter_bytes = split ? static_cast<size_t>(bg) * sizeof(unsigned int) : 0;
  return MQA_OK;
}

// The prefill kernel (several tokens, more than 64 rows per KV head): no scratch, no overlap.
int launch_prefill(const DecodePlan& p) {
  CUtensorMap tmk, tmv;
  if (!make_cache_map(&tmk, p.k_cache, static_cast<int>(p.bg), p.n_max, p.d_h, 2) ||
      !make_cache_map(&tmv, p.v_cache, static_cast<int>(p.bg), p.n_max, p.d_h, 2))
    return MQA_ERR_CUDA;
  DecodeParams P = {};
  P.q = reinterpret_cast<const __nv_bfloat16*>(p.q);
  P.seq_lens = p.seq_lens;
  P.out = reinterpret_cast<__nv_bfloat16*>(p.out);
  P.b = p.b;
  P.h = p.h;
  P.g = p.g;
  P.G = p.G;
  P.T = p.T;
  P.Gh = p.Gh;
  P.n_max = p.n_max;
  P.num_ctas = static_cast<int>(p.ctas);
  P.scale_log2 = p.scale * 1.4426950408889634f;
  P.kq_scale = P.vq_scale = P.out_scale = 1.f;
  P.timeout_ns = g_wait_limit_ns.load();
  P.drain_ns = kWaitLimitNs;
  P.debug_stall = g_debug_stall.load();
  P.early_writes = 0;
  AttnKernelChoice kc;
  kc.fn = p.d_h == 128 ? mqa::prefill_attention_tc_kernel<128> : mqa::prefill_attention_tc_kernel<64>;
  kc.threads = mqa::kTcThreads;
  kc.smem = mqa::pf_smem_bytes(p.d_h);
  if (int st = prepare_kernel(p.dev, kc, kc.smem)) return st;
  kc.fn<<<static_cast<unsigned>(p.ctas), kc.threads, kc.smem, p.stream>>>(tmk, tmv, P);
  g_launches.fetch_add(1);
  return launch_error();
}

// T new rows per sequence into contiguous bf16 caches (one 16-byte chunk per thread).
int launch_append_multi(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_cache,
                        mqa_bf16* v_cache, const int32_t* pos, int b, int T, int g, int d_h,
                        int n_max, cudaStream_t stream) {
  const long long rows = static_cast<long long>(b) * T * g;
  const int chunks = d_h / 8;
  const long long total = rows * chunks;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65535 ? want : 65535);
  mqa::kv_append_kernel<<<blocks, threads, 0, stream>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), pos, b, T, g, chunks,
      n_max);
  g_launches.fetch_add(1);
  return launch_error();
}

// `sc.clear`: zero the scratch's whole counter region first. The counters are zero whenever the
// scratch is fresh and every finished call leaves them at zero; only a call that gave up
// (MQA_ERR_TIMEOUT) can leave them dirty, and it may have used more of them than this call does.
int launch_decode(const DecodePlan& p, const Scratch& sc) {
  void* partials = sc.partials;
  unsigned int* counters = sc.counters;
  CUtensorMap tmk, tmv;
  if (p.paged.table) {
    const long long pages_g = static_cast<long long>(p.paged.num_pages) * p.g;
    if (!make_pool_map(&tmk, p.k_cache, pages_g, p.paged.page_size, p.d_h, p.eb) ||
        !make_pool_map(&tmv, p.v_cache, pages_g, p.paged.page_size, p.d_h, p.eb))
      return MQA_ERR_CUDA;
  } else if (!make_cache_map(&tmk, p.k_cache, static_cast<int>(p.bg), p.n_max, p.d_h, p.eb) ||
             !make_cache_map(&tmv, p.v_cache, static_cast<int>(p.bg), p.n_max, p.d_h, p.eb)) {
    return MQA_ERR_CUDA;
  }

  DecodeParams P;
  P.q = reinterpret_cast<const __nv_bfloat16*>(p.q);
  P.seq_lens = p.seq_lens;
  P.out = reinterpret_cast<__nv_bfloat16*>(p.out);
  P.part_o = static_cast<float*>(partials);
  P.part_ml = partials ? reinterpret_cast<float2*>(static_cast<char*>(partials) + p.part_o_bytes)
                       : nullptr;
  P.seg_arrivals = counters;
  if (counters && sc.clear &&
      cudaMemsetAsync(sc.counter_region, 0, sc.counter_region_bytes, p.stream) != cudaSuccess)
    return MQA_ERR_CUDA;
  P.b = p.b;
  P.h = p.h;
  P.g = p.g;
  P.G = p.G;
  P.T = p.T;
  P.Gh = p.Gh;
  P.n_max = p.n_max;
  P.num_ctas = static_cast<int>(p.ctas);
  // fp8: the logits are scale * k_scale * (q . codes); the output is v_scale * (P codes) / l
  P.scale_log2 = p.scale * (p.eb == 1 ? p.k_scale : 1.f) * 1.4426950408889634f;
  P.kq_scale = p.k_scale;
  P.vq_scale = p.v_scale;
  P.out_scale = p.eb == 1 ? p.v_scale : 1.f;
  P.timeout_ns = g_wait_limit_ns.load();
  P.drain_ns = kWaitLimitNs;
  P.debug_stall = g_debug_stall.load();
  P.pos = p.pos;
  P.k_new = reinterpret_cast<const uint4*>(p.k_new);
  P.v_new = reinterpret_cast<const uint4*>(p.v_new);
  // the caches are written only at the rows the fused append targets
  P.k_rows = p.pos ? reinterpret_cast<uint4*>(const_cast<mqa_bf16*>(p.k_cache)) : nullptr;
  P.v_rows = p.pos ? reinterpret_cast<uint4*>(const_cast<mqa_bf16*>(p.v_cache)) : nullptr;
  P.page_table = p.paged.table;
  P.page_size = p.paged.page_size;
  P.max_pages = p.paged.max_pages;
  P.num_pages = p.paged.num_pages;

  // fp8 caches: mma.sync at every group size unless forced. Measured on B300 (32K rows, launches
  // back to back): the fp8 CUDA-core consumer reaches 0.37 (G = 1) to 0.21 (G = 7) of the copy
  // bandwidth on fp8 bytes, the fp16 mma.sync consumer 0.72-0.73 at every G.
  const Path fp8_path = p.path_forced ? p.path : kPathMmaSync;
  const AttnKernelChoice kc = p.eb == 1       ? pick_kernel_fp8(fp8_path, p.G, p.b)
                              : p.d_h == 128 ? pick_kernel<128>(p.path, p.G, p.b, p.T)
                                             : pick_kernel<64>(p.path, p.G, p.b, p.T);
  if (!kc.fn) return MQA_ERR_UNSUPPORTED;
  if (p.paged.table && p.path == kPathTcgen05) return MQA_ERR_UNSUPPORTED;
  if (int st = prepare_kernel(p.dev, kc, kc.smem)) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.ctas));
  cfg.blockDim = dim3(static_cast<unsigned>(kc.threads));
  cfg.dynamicSmemBytes = kc.smem;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  const bool overlap = kc.pdl && overlap_on(p.dev, p.stream);
  if (overlap) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // early writes need scratch the launch ahead does not share: a workspace half, or none at all
  // (one CTA); the no-alloc array is a single region, so those launches wait before writing.
  // They also hold the next launch back until the launch two back has finished, which costs more
  // than it saves on launches that read much: only caches up to kEarlyWritesMaxCacheBytes take
  // them.
  const double cache_bytes = 2.0 * static_cast<double>(p.bg) * p.n_max * p.d_h * p.eb;
  P.early_writes =
      (overlap && (sc.alternating || p.ctas == 1) && cache_bytes <= kEarlyWritesMaxCacheBytes)
          ? 1
          : 0;
  if (cudaLaunchKernelEx(&cfg, kc.fn, tmk, tmv, P) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  g_launches.fetch_add(1);
  return launch_error();
}

// ------------------------------------------------------------------------------------------------
// Scratch for mqa_decode_attention_noalloc: a fixed array in this module's device memory, so the
// call itself allocates nothing. In host code the array's name is only a host-side stand-in, so
// its device address is looked up once per device (with that device current) and cached.
// ------------------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[MQA_NOALLOC_SCRATCH_BYTES];
// Its first kNoallocCounterBytes hold the per-segment arrival counters (MQA_NOALLOC_MAX_SEGMENTS
// of them); the split partial states follow.
constexpr size_t kNoallocCounterBytes = MQA_NOALLOC_MAX_SEGMENTS * sizeof(unsigned int);

struct NoallocScratch {
  void* ptr = nullptr;       // device address of g_noalloc_scratch on this device
  uint64_t clean_epoch = 0;  // the array starts zeroed, so its counters start clean
};
std::mutex g_noalloc_mutex;
std::map<int, NoallocScratch> g_noalloc_addr;  // device ordinal -> its copy of the array

int noalloc_scratch_address(int dev, Scratch* out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  auto it = g_noalloc_addr.find(dev);
  if (it == g_noalloc_addr.end()) {
    NoallocScratch sc;
    if (cudaGetSymbolAddress(&sc.ptr, g_noalloc_scratch) != cudaSuccess || sc.ptr == nullptr)
      return MQA_ERR_CUDA;
    sc.clean_epoch = g_timeout_epoch.load();
    it = g_noalloc_addr.emplace(dev, sc).first;
  }
  const uint64_t epoch = g_timeout_epoch.load();
  // the counters keep a fixed leading region of the array, so no other call's partial states
  // ever land on them; after a timeout that whole region is cleared
  out->clear = it->second.clean_epoch != epoch;
  it->second.clean_epoch = epoch;
  out->counters = static_cast<unsigned int*>(it->second.ptr);
  out->partials = static_cast<char*>(it->second.ptr) + kNoallocCounterBytes;
  out->counter_region = it->second.ptr;
  out->counter_region_bytes = kNoallocCounterBytes;
  out->alternating = false;
  return MQA_OK;
}

// T rows per sequence through a page table, bf16 (eb = 2) or fp8 codes (eb = 1), after the
// host checks of the paged calls.
int launch_append_paged_rows(const mqa_bf16* k_new, const mqa_bf16* v_new, void* k_pool,
                             void* v_pool, const int32_t* pos, const PagedCache& pg, int b, int T,
                             int g, int d_h, int eb, float k_scale, float v_scale,
                             cudaStream_t stream) {
  const long long rows = static_cast<long long>(b) * T * g;
  if (rows > (1ll << 31)) return MQA_ERR_UNSUPPORTED;
  const long long total = rows * (d_h * eb / 16);
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65535 ? want : 65535);
  auto kern = eb == 2 ? mqa::kv_append_paged_rows_kernel<2> : mqa::kv_append_paged_rows_kernel<1>;
  kern<<<blocks, threads, 0, stream>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), pos, pg.table, b, T, g, d_h,
      pg.page_size, pg.max_pages, pg.num_pages, k_scale, v_scale);
  g_launches.fetch_add(1);
  return launch_error();
}

// Host checks shared by the paged appends: pointers, alignment, sizes, the pool geometry.
int check_paged_append(const mqa_bf16* k_new, const mqa_bf16* v_new, const void* k_pool,
                       const void* v_pool, const int32_t* pos, const PagedCache& pg, int b, int T,
                       int g, int d_h) {
  if (!k_new || !v_new || !k_pool || !v_pool || !pos) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || T <= 0 || g <= 0 || d_h <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  int n_max = 0;
  if (int st = check_paged(pg, g, d_h, &n_max)) return st;
  if (d_h != 64 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  return MQA_OK;
}

PagedCache paged_cache(const int32_t* table, int page_size, int max_pages, int num_pages) {
  PagedCache pg;
  pg.table = table;
  pg.page_size = page_size;
  pg.max_pages = max_pages;
  pg.num_pages = num_pages;
  return pg;
}

// Paged attention (and the fused step when k_new is given) after the host checks: fp8 codes
// (eb = 1, with scales) or bf16 (eb = 2), T tokens per sequence on the decode kernels.
int paged_decode(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                 const void* k_pool, const void* v_pool, const int32_t* pos,
                 const PagedCache& pg, const int32_t* seq_lens, mqa_bf16* out, int b, int T,
                 int h, int g, int d_h, float scale, int eb, float k_scale, float v_scale,
                 void* stream) {
  if (g <= 0) return MQA_ERR_INVALID_ARG;
  if (k_new && (!v_new || !pos)) return MQA_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new) ||
                (reinterpret_cast<uintptr_t>(pos) & 3u)))
    return MQA_ERR_INVALID_ARG;
  if (eb == 1 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f &&
                   v_scale > 0.f))
    return MQA_ERR_INVALID_ARG;
  if (eb == 1 && d_h > 0 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  int n_max = 0;
  if (int st = check_paged(pg, g, d_h, &n_max)) return st;
  DecodePlan plan;
  if (int st = plan_decode(q, static_cast<const mqa_bf16*>(k_pool),
                           static_cast<const mqa_bf16*>(v_pool), seq_lens, out, b, h, g, d_h,
                           n_max, scale, stream, &plan, T))
    return st;
  if (plan.prefill) return MQA_ERR_UNSUPPORTED;  // the prefill kernel reads contiguous caches
  plan.paged = pg;
  plan.eb = eb;
  plan.k_scale = eb == 1 ? k_scale : 1.f;
  plan.v_scale = eb == 1 ? v_scale : 1.f;
  plan.k_new = k_new;
  plan.v_new = v_new;
  plan.pos = pos;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

}  // namespace

extern "C" {

const char* mqa_status_string(int status) {
  switch (status) {
    case MQA_OK: return "MQA_OK";
    case MQA_ERR_INVALID_ARG: return "MQA_ERR_INVALID_ARG: invalid argument";
    case MQA_ERR_UNSUPPORTED: return "MQA_ERR_UNSUPPORTED: shape or setting not supported";
    case MQA_ERR_CUDA: return "MQA_ERR_CUDA: CUDA runtime error";
    case MQA_ERR_DEVICE_BOUNDS:
      return "MQA_ERR_DEVICE_BOUNDS: a pos, seq_lens or page-table entry out of range";
    case MQA_ERR_TIMEOUT: return "MQA_ERR_TIMEOUT: an in-kernel wait timed out";
    default: return "unknown mqa status";
  }
}

uint64_t mqa_kernel_launch_count(void) { return g_launches.load(); }

int mqa_debug_override(int num_ctas, int path) {
  if (num_ctas < 0 || path < 0 || path > 3) return MQA_ERR_INVALID_ARG;
  g_force_ctas.store(num_ctas);
  g_force_path.store(path);
  return MQA_OK;
}

int mqa_get_device_status(void* stream, int* status_out) {
  if (!status_out) return MQA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MQA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, mqa::g_device_status, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MQA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(mqa::g_device_status, &zero, sizeof(int), 0,
                              cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MQA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MQA_ERR_CUDA;
  if (v == MQA_ERR_TIMEOUT) g_timeout_epoch.fetch_add(1);
  *status_out = v;
  return MQA_OK;
}

int mqa_set_launch_overlap(void* stream, int on) {
  if (on != 0 && on != 1) return MQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_overlap_mutex);
  g_overlap[{dev, reinterpret_cast<uintptr_t>(stream)}] = on != 0;
  return MQA_OK;
}

int mqa_debug_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kWaitLimitNs : ns);
  return MQA_OK;
}

int mqa_debug_stall(int on) {
  if (on < 0 || on > 2) return MQA_ERR_INVALID_ARG;
  g_debug_stall.store(on);
  return MQA_OK;
}

int mqa_debug_timeout_site(int* site_out) {
  if (!site_out) return MQA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MQA_ERR_CUDA;
  int v[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(v, mqa::g_timeout_site, sizeof(v)) != cudaSuccess) return MQA_ERR_CUDA;
  const int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(mqa::g_timeout_site, zero, sizeof(zero)) != cudaSuccess)
    return MQA_ERR_CUDA;
  for (int i = 0; i < 4; ++i) site_out[i] = v[i];
  return MQA_OK;
}

int mqa_kv_append(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_cache,
                  mqa_bf16* v_cache, const int32_t* pos, int b, int g, int d_h, int n_max,
                  void* stream) {
  // ---- host checks (no CUDA call before this block is done) ----
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(b) * g;
  if (rows > (1ll << 31) || static_cast<double>(rows) * n_max * d_h > 9.0e18)
    return MQA_ERR_UNSUPPORTED;

  const int chunks = d_h / 8;
  const long long total = rows * chunks;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65535 ? want : 65535);
  mqa::kv_append_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), pos, b, 1, g, chunks,
      n_max);
  g_launches.fetch_add(1);
  return launch_error();
}

int mqa_decode_attention(const mqa_bf16* q, const mqa_bf16* k_cache, const mqa_bf16* v_cache,
                         const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h,
                         int n_max, float scale, void* stream) {
  DecodePlan plan;
  if (int st = plan_decode(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan))
    return st;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_decode_step(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                    mqa_bf16* k_cache, mqa_bf16* v_cache, const int32_t* pos,
                    const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h,
                    int n_max, float scale, void* stream) {
  if (!k_new || !v_new || !pos) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  DecodePlan plan;
  if (int st = plan_decode(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan))
    return st;
  plan.k_new = k_new;
  plan.v_new = v_new;
  plan.pos = pos;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_kv_append_paged(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_pool,
                        mqa_bf16* v_pool, const int32_t* pos, const int32_t* page_table, int b,
                        int g, int d_h, int page_size, int max_pages, int num_pages,
                        void* stream) {
  // ---- host checks (no CUDA call before this block is done) ----
  if (!k_new || !v_new || !k_pool || !v_pool || !pos) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  PagedCache pg;
  pg.table = page_table;
  pg.page_size = page_size;
  pg.max_pages = max_pages;
  pg.num_pages = num_pages;
  int n_max = 0;
  if (int st = check_paged(pg, g, d_h, &n_max)) return st;
  if (d_h != 64 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(b) * g;
  if (rows > (1ll << 31)) return MQA_ERR_UNSUPPORTED;

  const int chunks = d_h / 8;
  const long long total = rows * chunks;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65535 ? want : 65535);
  mqa::kv_append_paged_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), pos, page_table, b, g,
      chunks, page_size, max_pages, num_pages);
  g_launches.fetch_add(1);
  return launch_error();
}

int mqa_decode_attention_paged(const mqa_bf16* q, const mqa_bf16* k_pool, const mqa_bf16* v_pool,
                               const int32_t* page_table, const int32_t* seq_lens, mqa_bf16* out,
                               int b, int h, int g, int d_h, int page_size, int max_pages,
                               int num_pages, float scale, void* stream) {
  if (g <= 0) return MQA_ERR_INVALID_ARG;
  PagedCache pg;
  pg.table = page_table;
  pg.page_size = page_size;
  pg.max_pages = max_pages;
  pg.num_pages = num_pages;
  int n_max = 0;
  if (int st = check_paged(pg, g, d_h, &n_max)) return st;
  DecodePlan plan;
  if (int st = plan_decode(q, k_pool, v_pool, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan))
    return st;
  plan.paged = pg;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_decode_step_paged(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                          mqa_bf16* k_pool, mqa_bf16* v_pool, const int32_t* pos,
                          const int32_t* page_table, const int32_t* seq_lens, mqa_bf16* out,
                          int b, int h, int g, int d_h, int page_size, int max_pages,
                          int num_pages, float scale, void* stream) {
  if (!k_new || !v_new || !pos || g <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  PagedCache pg;
  pg.table = page_table;
  pg.page_size = page_size;
  pg.max_pages = max_pages;
  pg.num_pages = num_pages;
  int n_max = 0;
  if (int st = check_paged(pg, g, d_h, &n_max)) return st;
  DecodePlan plan;
  if (int st = plan_decode(q, k_pool, v_pool, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan))
    return st;
  plan.paged = pg;
  plan.k_new = k_new;
  plan.v_new = v_new;
  plan.pos = pos;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

// fp8 caches: the scales must be finite and positive; the kernels read d_h = 128 rows.
static bool valid_fp8_scales(float k_scale, float v_scale) {
  return std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f;
}

int mqa_kv_append_fp8(const mqa_bf16* k_new, const mqa_bf16* v_new, uint8_t* k_cache,
                      uint8_t* v_cache, const int32_t* pos, int b, int g, int d_h, int n_max,
                      float k_scale, float v_scale, void* stream) {
  // ---- host checks (no CUDA call before this block is done) ----
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  if (!valid_fp8_scales(k_scale, v_scale)) return MQA_ERR_INVALID_ARG;
  if (d_h != 128) return MQA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(b) * g;
  if (rows > (1ll << 31) || static_cast<double>(rows) * n_max * d_h > 9.0e18)
    return MQA_ERR_UNSUPPORTED;

  const long long total = rows * (d_h / 16);
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65535 ? want : 65535);
  mqa::kv_append_fp8_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), pos, b, g, d_h, n_max,
      k_scale, v_scale);
  g_launches.fetch_add(1);
  return launch_error();
}

int mqa_decode_attention_fp8(const mqa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g,
                             int d_h, int n_max, float scale, float k_scale, float v_scale,
                             void* stream) {
  if (!valid_fp8_scales(k_scale, v_scale)) return MQA_ERR_INVALID_ARG;
  if (d_h > 0 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (int st = plan_decode(q, reinterpret_cast<const mqa_bf16*>(k_cache),
                           reinterpret_cast<const mqa_bf16*>(v_cache), seq_lens, out, b, h, g,
                           d_h, n_max, scale, stream, &plan))
    return st;
  plan.eb = 1;
  plan.k_scale = k_scale;
  plan.v_scale = v_scale;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_decode_step_fp8(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                        uint8_t* k_cache, uint8_t* v_cache, const int32_t* pos,
                        const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g, int d_h,
                        int n_max, float scale, float k_scale, float v_scale, void* stream) {
  if (!k_new || !v_new || !pos) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  if (!valid_fp8_scales(k_scale, v_scale)) return MQA_ERR_INVALID_ARG;
  if (d_h > 0 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (int st = plan_decode(q, reinterpret_cast<const mqa_bf16*>(k_cache),
                           reinterpret_cast<const mqa_bf16*>(v_cache), seq_lens, out, b, h, g,
                           d_h, n_max, scale, stream, &plan))
    return st;
  plan.eb = 1;
  plan.k_scale = k_scale;
  plan.v_scale = v_scale;
  plan.k_new = k_new;
  plan.v_new = v_new;
  plan.pos = pos;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_kv_append_multi(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_cache,
                        mqa_bf16* v_cache, const int32_t* pos, int b, int T, int g, int d_h,
                        int n_max, void* stream) {
  // ---- host checks (no CUDA call before this block is done) ----
  if (!k_new || !v_new || !k_cache || !v_cache || !pos) return MQA_ERR_INVALID_ARG;
  if (b <= 0 || T <= 0 || g <= 0 || d_h <= 0 || n_max <= 0) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return MQA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(b) * T * g;
  if (rows > (1ll << 31) || static_cast<double>(b) * g * n_max * d_h > 9.0e18)
    return MQA_ERR_UNSUPPORTED;

  return launch_append_multi(k_new, v_new, k_cache, v_cache, pos, b, T, g, d_h, n_max,
                             static_cast<cudaStream_t>(stream));
}

int mqa_decode_attention_multi(const mqa_bf16* q, const mqa_bf16* k_cache,
                               const mqa_bf16* v_cache, const int32_t* seq_lens, mqa_bf16* out,
                               int b, int T, int h, int g, int d_h, int n_max, float scale,
                               void* stream) {
  DecodePlan plan;
  if (int st = plan_decode(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan, T))
    return st;
  if (plan.prefill) return launch_prefill(plan);
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_decode_step_multi(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                          mqa_bf16* k_cache, mqa_bf16* v_cache, const int32_t* pos,
                          const int32_t* seq_lens, mqa_bf16* out, int b, int T, int h, int g,
                          int d_h, int n_max, float scale, void* stream) {
  if (!k_new || !v_new || !pos) return MQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MQA_ERR_INVALID_ARG;
  DecodePlan plan;
  if (int st = plan_decode(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan, T))
    return st;
  if (plan.prefill) {
    // every unit of a sequence reads its T new rows: append them first, then attend
    if (int st = launch_append_multi(k_new, v_new, k_cache, v_cache, pos, b, T, g, d_h, n_max,
                                     plan.stream))
      return st;
    return launch_prefill(plan);
  }
  plan.k_new = k_new;
  plan.v_new = v_new;
  plan.pos = pos;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = get_workspace(plan.dev, plan.stream, plan.partial_bytes, plan.counter_bytes, &sc))
      return st;
  }
  return launch_decode(plan, sc);
}

int mqa_decode_attention_noalloc(const mqa_bf16* q, const mqa_bf16* k_cache,
                                 const mqa_bf16* v_cache, const int32_t* seq_lens, mqa_bf16* out,
                                 int b, int h, int g, int d_h, int n_max, float scale,
                                 void* stream) {
  DecodePlan plan;
  if (int st = plan_decode(q, k_cache, v_cache, seq_lens, out, b, h, g, d_h, n_max, scale, stream,
                           &plan))
    return st;
  if (plan.counter_bytes > kNoallocCounterBytes ||
      plan.partial_bytes > MQA_NOALLOC_SCRATCH_BYTES - kNoallocCounterBytes)
    return MQA_ERR_UNSUPPORTED;
  Scratch sc;
  if (plan.ctas > 1) {
    if (int st = noalloc_scratch_address(plan.dev, &sc)) return st;
  }
  return launch_decode(plan, sc);
}

int mqa_kv_append_paged_multi(const mqa_bf16* k_new, const mqa_bf16* v_new, mqa_bf16* k_pool,
                              mqa_bf16* v_pool, const int32_t* pos, const int32_t* page_table,
                              int b, int T, int g, int d_h, int page_size, int max_pages,
                              int num_pages, void* stream) {
  const PagedCache pg = paged_cache(page_table, page_size, max_pages, num_pages);
  if (int st = check_paged_append(k_new, v_new, k_pool, v_pool, pos, pg, b, T, g, d_h)) return st;
  return launch_append_paged_rows(k_new, v_new, k_pool, v_pool, pos, pg, b, T, g, d_h, 2, 1.f,
                                  1.f, static_cast<cudaStream_t>(stream));
}

int mqa_decode_attention_paged_multi(const mqa_bf16* q, const mqa_bf16* k_pool,
                                     const mqa_bf16* v_pool, const int32_t* page_table,
                                     const int32_t* seq_lens, mqa_bf16* out, int b, int T, int h,
                                     int g, int d_h, int page_size, int max_pages, int num_pages,
                                     float scale, void* stream) {
  return paged_decode(q, nullptr, nullptr, k_pool, v_pool, nullptr,
                      paged_cache(page_table, page_size, max_pages, num_pages), seq_lens, out, b,
                      T, h, g, d_h, scale, 2, 1.f, 1.f, stream);
}

int mqa_decode_step_paged_multi(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                                mqa_bf16* k_pool, mqa_bf16* v_pool, const int32_t* pos,
                                const int32_t* page_table, const int32_t* seq_lens,
                                mqa_bf16* out, int b, int T, int h, int g, int d_h, int page_size,
                                int max_pages, int num_pages, float scale, void* stream) {
  if (!k_new) return MQA_ERR_INVALID_ARG;
  return paged_decode(q, k_new, v_new, k_pool, v_pool, pos,
                      paged_cache(page_table, page_size, max_pages, num_pages), seq_lens, out, b,
                      T, h, g, d_h, scale, 2, 1.f, 1.f, stream);
}

int mqa_kv_append_paged_fp8(const mqa_bf16* k_new, const mqa_bf16* v_new, uint8_t* k_pool,
                            uint8_t* v_pool, const int32_t* pos, const int32_t* page_table, int b,
                            int g, int d_h, int page_size, int max_pages, int num_pages,
                            float k_scale, float v_scale, void* stream) {
  const PagedCache pg = paged_cache(page_table, page_size, max_pages, num_pages);
  if (int st = check_paged_append(k_new, v_new, k_pool, v_pool, pos, pg, b, 1, g, d_h)) return st;
  if (!valid_fp8_scales(k_scale, v_scale)) return MQA_ERR_INVALID_ARG;
  if (d_h != 128) return MQA_ERR_UNSUPPORTED;
  return launch_append_paged_rows(k_new, v_new, k_pool, v_pool, pos, pg, b, 1, g, d_h, 1, k_scale,
                                  v_scale, static_cast<cudaStream_t>(stream));
}

int mqa_decode_attention_paged_fp8(const mqa_bf16* q, const uint8_t* k_pool,
                                   const uint8_t* v_pool, const int32_t* page_table,
                                   const int32_t* seq_lens, mqa_bf16* out, int b, int h, int g,
                                   int d_h, int page_size, int max_pages, int num_pages,
                                   float scale, float k_scale, float v_scale, void* stream) {
  return paged_decode(q, nullptr, nullptr, k_pool, v_pool, nullptr,
                      paged_cache(page_table, page_size, max_pages, num_pages), seq_lens, out, b,
                      1, h, g, d_h, scale, 1, k_scale, v_scale, stream);
}

int mqa_decode_step_paged_fp8(const mqa_bf16* q, const mqa_bf16* k_new, const mqa_bf16* v_new,
                              uint8_t* k_pool, uint8_t* v_pool, const int32_t* pos,
                              const int32_t* page_table, const int32_t* seq_lens, mqa_bf16* out,
                              int b, int h, int g, int d_h, int page_size, int max_pages,
                              int num_pages, float scale, float k_scale, float v_scale,
                              void* stream) {
  if (!k_new) return MQA_ERR_INVALID_ARG;
  return paged_decode(q, k_new, v_new, k_pool, v_pool, pos,
                      paged_cache(page_table, page_size, max_pages, num_pages), seq_lens, out, b,
                      1, h, g, d_h, scale, 1, k_scale, v_scale, stream);
}

}  // extern "C"
