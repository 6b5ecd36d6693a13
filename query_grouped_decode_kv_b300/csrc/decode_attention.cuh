// decode_attention.cuh -- grouped decode attention for sm_103a.
//
// Definition ("分组查询注意力（GQA）与多查询注意力（MQA）深度实战", ybb.press, §五): for query head i
// of sequence bi, with j = i / G and G = h / g,
//     O_i = sum_{t < L} softmax_t(scale * q_i . K_{j,t}) V_{j,t},   L = seq_lens[bi].
//
// Work decomposition. The unit of work is a tile of kTileKeys consecutive cache rows of one
// "segment" (sequence bi, KV head j). Segments are laid end to end in (bi, j) order, forming
// W = g * sum_bi ceil(L_bi / kTileKeys) tiles, and CTA c of P takes the contiguous tile range
// [c*W/P, (c+1)*W/P). Lengths live on the device, so every CTA derives W and its range from
// seq_lens itself: the split is balanced to within one tile whatever the length mix, and the host
// never synchronises to read lengths. A segment that lies entirely inside one CTA's range is
// finished by that CTA; otherwise each CTA writes a partial softmax state (m, l, o) into slot
// c + segment and counts its arrival on the segment's counter, and the last CTA to arrive merges
// the slots with the log-sum-exp identity (then resets the counter to zero for the next call).
//
// Inside a CTA: two producer warps stream alternate tiles' K and V rows from HBM into a ring of
// shared-memory stages with bulk tensor copies (TMA, 128-byte swizzle); four or eight consumer
// warps read every stage once, so the K/V bytes of a KV head are fetched exactly once and reused
// by all G query heads that share them. Each consumer warp keeps an online softmax (running max m
// and sum l in fp32, log2 domain) for its slice of the tile's keys; at a segment's end the warps'
// states are combined through shared memory.
//
// Inner products: the grouped heads run on tensor cores in mma.sync m16n8k16 products (fp32
// accumulate): up to 8 heads as the N columns of transposed products (S^T = K q^T, then
// O^T += V^T P^T), beyond that as the M rows (S = Q K^T, then O += P V). With one or two heads per
// K/V row (MHA-like grouping) CUDA cores do fp32 FMAs instead; they serve up to seven heads when
// forced.
//
// Every wait is bounded in time: on expiry the kernel latches MQA_ERR_TIMEOUT and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "status.cuh"

namespace mqa {

constexpr int kTileKeys = 64;       // cache rows per pipeline stage
constexpr int kRingBytes = 128 * 1024;  // the shared-memory ring of K/V stages
constexpr int kSwizzleRowBytes = 128;
constexpr uint32_t kOnesBf16x2 = 0x3F803F80u;  // two bf16 ones (the B fragment of P 1)
constexpr uint32_t kOnesF16x2 = 0x3C003C00u;   // two fp16 ones
// NW (a template parameter below) is the number of consumer warps: 4 or 8.
//  - NW = 4: a producer warp, a launch-order warp and a second producer warp come on top
//    (224 threads).
//  - NW = 8: two consumer warpgroups and one producer warpgroup (384 threads). The launch gives
//    every thread kLaunchRegsWide registers (the most 384 threads can have on one SM); the
//    producer warpgroup then hands registers back (setmaxnreg.dec to kProducerRegs) and the
//    consumer warpgroups take them (setmaxnreg.inc to kConsumerRegs). Warp NW is the producer,
//    warp NW + 1 the launch-order warp, warp NW + 2 the second producer.
// The launch-order warp (warp NW + 1) matters for launches that overlap the kernel ahead of them
// on the stream: its lane 0 waits for that kernel to finish and only then lets the next launch be
// scheduled, so that a launch never starts before the one two back has finished.
__host__ __device__ constexpr int threads_of(int NW) { return NW == 8 ? 384 : 32 * (NW + 3); }
// Producer warps (warps NW and NW + 2, alternate tiles). Measured on B300 against one producer
// warp, launches back to back: the 70B-class layer over fp8 codes 62.1-62.7 us against 68.7 us
// contiguous, 8-row fp8 pages 0.69 of the copy bandwidth against 0.42; the 80-layer bf16 step
// 7,835 against 7,913 us; mha_ref 152.5 against 157.7 us.
constexpr int kPagedProducers = 2;       // over paged caches
constexpr int kContiguousProducers = 2;  // over contiguous caches
constexpr int kLaunchRegsWide = 168;
constexpr int kProducerRegs = 72;
constexpr int kConsumerRegs = 216;
static_assert(2 * 128 * kConsumerRegs + 128 * kProducerRegs <= 384 * kLaunchRegsWide,
              "the register split must fit in what the launch allocated");
static_assert(2 * 32 * kConsumerRegs + 32 * kProducerRegs <= 16384,
              "two consumer warps and one producer warp share a sub-partition's registers");
constexpr int kMaxBatch = 8192;
constexpr int kMaxGroup = 64;       // largest G = h / g served
constexpr int kMaxCcHeads = 7;      // the CUDA-core consumers serve G < 8
constexpr int kCcWarpKeys = 16;     // keys per warp and tile in the CUDA-core consumer
constexpr float kLazyLog2 = 8.f;    // softmax reference slack (log2 units), see MmaConsumer::tile

struct DecodeParams {
  const __nv_bfloat16* q;     // [b][T][h][D]
  const int32_t* seq_lens;    // [b]
  __nv_bfloat16* out;         // [b][T][h][D]
  float* part_o;              // [slots][G][D]   un-normalised partial outputs
  float2* part_ml;            // [slots][G]      (running max in log2 units, running sum)
  unsigned int* seg_arrivals; // [b*g] CTAs that have stored a partial; zero between calls
  // A segment (sequence bi, KV head j) has G = T * Gh rows: the Gh query heads of the group for
  // each of the T new tokens, row r = t * Gh + hh. Token t attends the first L - T + 1 + t rows of
  // the cache (causal); with T = 1 a row is a head and every row attends all L rows.
  int b, h, g, G, n_max;
  int T, Gh;
  int num_ctas;               // P
  float scale_log2;           // scale * log2(e)
  unsigned long long timeout_ns;  // limit of every in-kernel wait
  unsigned long long drain_ns;    // limit of the waits for a CTA's own work in flight at exit
  int debug_stall;                // testing: consumers wait on a barrier nothing completes,
                                  // 1: before their first tile; 2: right after counting their
                                  // first arrival at a split segment (before any merge)
  // Fused append (mqa_decode_step): this step's K/V rows, token t written at row pos[bi] + t of
  // the caches before any tile holding that row is loaded. All null when the call only attends.
  const int32_t* pos;         // [b]
  const uint4* k_new;         // [b][T][g][D/8] 16-byte chunks
  const uint4* v_new;
  uint4* k_rows;              // the caches as 16-byte chunks, [b][g][n_max][D/8]
  uint4* v_rows;
  // Paged caches (all null / zero for contiguous ones): the caches are pools of pages
  // [num_pages][g][page_size][D], and row t of sequence bi lives in page
  // page_table[bi][t / page_size] at row t % page_size; n_max = max_pages * page_size.
  const int32_t* page_table;  // [b][max_pages]
  int page_size, max_pages, num_pages;
  // fp8 caches: the fused append stores e4m3(x / kq_scale) (and V with vq_scale); every final
  // output is multiplied by out_scale (the V scale; 1 for bf16 caches, where it changes nothing)
  float kq_scale, vq_scale, out_scale;
  // Launch overlap (programmatic dependent launch), for launches that may start while the kernel
  // ahead of them on the stream still runs. In both modes one thread per CTA waits
  // (griddepcontrol.wait) for that kernel and only then signals the dependents, so the next
  // launch starts only once the kernel ahead has finished: a launch never runs beside the one two
  // back, which may write its inputs and shares its half of the workspace. 0: the kernel also
  // waits before its first global write. 1 (early writes): the host gave this launch scratch that
  // the launch ahead does not use (the two halves of the workspace alternate) and the caller
  // guarantees that the launch ahead neither reads nor writes this launch's outputs, so the
  // writes do not wait.
  int early_writes;
};

// Stage geometry for head dimension D stored with EB bytes per element (2: bf16; 1: fp8 E4M3
// codes). A cache row is D * EB bytes, split into 128-byte swizzle rows ("halves"), one TMA box
// column range each; a stage holds one tile's K rows then its V rows; the ring holds kRingBytes,
// so the narrower rows get twice the stages (and twice the tiles in flight).
template <int D, int EB, int RB = kRingBytes>
struct Geometry {
  static constexpr int kRowBytes = D * EB;
  static constexpr int kHalves = kRowBytes / kSwizzleRowBytes;
  static constexpr int kBoxCols = kSwizzleRowBytes / EB;   // elements per 128-byte box row
  static constexpr int kKvBytes = kTileKeys * kRowBytes;   // one tile of K (or of V)
  static constexpr int kStageBytes = 2 * kKvBytes;
  static constexpr int kStages = RB / kStageBytes;  // in a 128 KB ring: 4 (32 KB stages) or 8
  static_assert(kRowBytes % kSwizzleRowBytes == 0 && kStages >= 2 && kStages <= 8, "geometry");
};

__host__ __device__ constexpr int comb_row_floats(int D) { return D + 8; }

// q of a segment in fp32 for the CUDA-core consumer: head hh's columns at hh * (D + 8), the upper
// half of them 4 floats further on, so that the two half-warps' same-address reads of the two
// halves land in different banks.
__host__ __device__ constexpr int cc_q_row_floats(int D) { return D + 8; }
__host__ __device__ constexpr int cc_q_index(int D, int hh, int d) {
  return hh * cc_q_row_floats(D) + d + (d >= D / 2 ? 4 : 0);
}

// Dynamic shared memory: [align pad][stages][comb_o][comb_ml][barriers][abort, merge flags]
// [page slots]. CR = rows per warp in the combine scratch (the head rows one consumer warp holds).
template <int D, int EB, int RB = kRingBytes>
__host__ __device__ constexpr int smem_fixed_bytes(int NW, int CR) {
  using Geo = Geometry<D, EB, RB>;
  return Geo::kStages * Geo::kStageBytes + NW * CR * comb_row_floats(D) * 4 + NW * CR * 8 +
         (2 * Geo::kStages + 2) * 8 + 16 +  // full, empty, cbar, stall; abort, merge flags
         kPagedProducers * 32 * 4 +         // the paged producers' looked-up pages
         kMaxCcHeads * cc_q_row_floats(D) * 4 +  // q of the segment in fp32 (CUDA-core consumer)
         NW * kMaxCcHeads * kCcWarpKeys * 4;     // its key weights, per warp
}
template <int D, int EB, int RB = kRingBytes>
__host__ __device__ constexpr size_t smem_bytes(int NW, int CR) {
  return 1024 + static_cast<size_t>(smem_fixed_bytes<D, EB, RB>(NW, CR));
}

// Element offset of row r (= t * Gh + hh) of segment (bi, j) in q or out ([b][T][h][D]).
// (One token: row r is head j * Gh + r, no division; the combine and merge loops call this per
// element.)
__device__ __forceinline__ size_t row_offset(const DecodeParams& P, int bi, int j, int r, int D) {
  if (P.T == 1) return (static_cast<size_t>(bi) * P.h + static_cast<size_t>(j) * P.Gh + r) * D;
  const int t = r / P.Gh, hh = r - t * P.Gh;
  return ((static_cast<size_t>(bi) * P.T + t) * P.h + static_cast<size_t>(j) * P.Gh + hh) * D;
}

// Rows of the cache that row r of a segment does not see, relative to the sequence's last
// token: T - 1 - t (0 with one token); padding rows (r >= G) see nothing.
__device__ __forceinline__ int row_lag(const DecodeParams& P, int r) {
  if (r >= P.G) return 0x7FFF;  // more than any tile: every key masked
  return P.T == 1 ? 0 : P.T - 1 - r / P.Gh;
}

// Tiles of a sequence of length L (0 when L is out of range: below the T new tokens, or past
// n_max).
__device__ __forceinline__ int tiles_of_length(int L, int n_max, int T) {
  return (L >= T && L >= 1 && L <= n_max) ? (L + kTileKeys - 1) / kTileKeys : 0;
}

// Byte offset of (key row, byte column c) inside one K or V stage: the row is split into halves
// of 128 bytes (one TMA box each); inside a half the 16-byte chunk index is XORed with (row % 8),
// the 128-byte swizzle the TMA applies. `c` must be a multiple of 16 here.
__device__ __forceinline__ uint32_t swz_bytes(uint32_t base, int key, int c) {
  const int half = c >> 7;
  const int chunk = (c >> 4) & 7;
  return base + static_cast<uint32_t>(half * (kTileKeys * kSwizzleRowBytes) +
                                      key * kSwizzleRowBytes + ((chunk ^ (key & 7)) << 4));
}
// The same for a bf16 stage and element column d (a multiple of 8).
__device__ __forceinline__ uint32_t swz(uint32_t base, int key, int d) {
  return swz_bytes(base, key, d * 2);
}

// ---------------------------------------------------------------------------------------------
// Fused append. Row pos[bi] of segment (bi, j) receives k_new[bi][j] and v_new[bi][j]. When a
// tile of the segment holds that row (pos < tiles * kTileKeys), the CTA that loads the tile writes
// the row first (write_new_row, from its producer warp, ordered before the tile's bulk copy by a
// generic-to-async proxy fence), so attention sees the new row. Every other valid row is written
// by append_uncovered_rows, spread over all CTAs; no tile of this launch reads it.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ bool row_is_loaded(int p, int L, int n_max, int T) {
  return static_cast<long long>(p) <
         static_cast<long long>(tiles_of_length(L, n_max, T)) * kTileKeys;
}

// First 16-byte chunk of cache row p of segment (bi, j) in the caches seen as chunks, or -1 when
// the page holding the row is out of range (paged caches; the row is then not written).
__device__ __forceinline__ long long row_chunk(const DecodeParams& P, int bi, int j, int p,
                                               int CH) {
  if (P.page_table == nullptr)
    return ((static_cast<long long>(bi) * P.g + j) * P.n_max + p) * CH;
  const int page = __ldg(P.page_table + static_cast<size_t>(bi) * P.max_pages + p / P.page_size);
  if (page < 0 || page >= P.num_pages) return -1;
  return ((static_cast<long long>(page) * P.g + j) * P.page_size + p % P.page_size) * CH;
}

// 16-byte chunk c of the cache row written for source row `src` (D bf16 values as 16-byte
// chunks): a copy for bf16 caches; for fp8 caches the codes e4m3(x / scale) of the 16 values
// x = src[16c .. 16c + 15], the division rounded once in fp32 (IEEE).
template <int EB>
__device__ __forceinline__ uint4 new_row_chunk(const uint4* src, int c, float scale) {
  if constexpr (EB == 2) {
    return __ldg(src + c);
  } else {
    const uint4 a = __ldg(src + 2 * c), b = __ldg(src + 2 * c + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t q[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[2 * i + k]);
        q[k] = f32x2_to_e4m3x2(__fdiv_rn(__low2float(x), scale),
                               __fdiv_rn(__high2float(x), scale));
      }
      out[i] = q[0] | (q[1] << 16);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
  }
}

template <int D, int EB>
__device__ __forceinline__ void append_uncovered_rows(const DecodeParams& P, int nthreads) {
  constexpr int CH = D * EB / 16;  // 16-byte chunks per cache row
  constexpr int CS = D / 8;        // 16-byte chunks per source row (bf16)
  const int T = P.T;
  const long long total = static_cast<long long>(P.b) * T * P.g * CH;
  const long long stride = static_cast<long long>(P.num_ctas) * nthreads;
  for (long long idx = static_cast<long long>(blockIdx.x) * nthreads + threadIdx.x; idx < total;
       idx += stride) {
    const long long src_row = idx / CH;  // = (bi * T + t) * g + j, the row of k_new / v_new
    const int c = static_cast<int>(idx - src_row * CH);
    const long long bt = src_row / P.g;
    const int j = static_cast<int>(src_row - bt * P.g);
    const int bi = static_cast<int>(bt / T);
    const int t = static_cast<int>(bt - static_cast<long long>(bi) * T);
    const int p0 = __ldg(P.pos + bi);
    if (p0 < 0 || static_cast<long long>(p0) + T > P.n_max) {
      if (c == 0 && t == 0 && j == 0) latch_status(kStatusDeviceBounds);
      continue;
    }
    const int p = p0 + t;
    if (row_is_loaded(p, __ldg(P.seq_lens + bi), P.n_max, T)) continue;
    const long long dst = row_chunk(P, bi, j, p, CH);
    if (dst < 0) {
      if (c == 0) latch_status(kStatusDeviceBounds);
      continue;
    }
    if (!P.early_writes) pdl_wait();  // else the launch ahead does not touch this row
    P.k_rows[dst + c] = new_row_chunk<EB>(P.k_new + src_row * CS, c, P.kq_scale);
    P.v_rows[dst + c] = new_row_chunk<EB>(P.v_new + src_row * CS, c, P.vq_scale);
  }
}

// One warp writes the K and V row of token t of segment (bi, j) at cache row `p` (lane = 16-byte
// chunk of the cache row).
template <int D, int EB>
__device__ __forceinline__ void write_new_row(const DecodeParams& P, int bi, int j, int t, int p,
                                              int lane) {
  constexpr int CH = D * EB / 16;
  constexpr int CS = D / 8;
  const long long src = ((static_cast<long long>(bi) * P.T + t) * P.g + j) * CS;
  const long long dst = row_chunk(P, bi, j, p, CH);
  if (dst < 0) {
    if (lane == 0) latch_status(kStatusDeviceBounds);
    return;
  }
  if (lane < CH) P.k_rows[dst + lane] = new_row_chunk<EB>(P.k_new + src, lane, P.kq_scale);
  else if (lane < 2 * CH)
    P.v_rows[dst + lane - CH] = new_row_chunk<EB>(P.v_new + src, lane - CH, P.vq_scale);
}

// The new rows of segment (bi, j) that tile `tile` holds ([p0, p0 + T) meets the tile's rows),
// written by the whole warp before the tile's copy; the caller fences and syncs the warp. Unless
// the launch has early writes, the writes wait for the kernel ahead on the stream to finish
// (programmatic dependent launch): that kernel may still be reading the rows being replaced.
template <int D, int EB>
__device__ __forceinline__ bool write_tile_rows(const DecodeParams& P, int bi, int j, int tile,
                                                int p0, int lane) {
  const int lo = max(p0, tile * kTileKeys), hi = min(p0 + P.T, (tile + 1) * kTileKeys);
  if (lo >= hi) return false;
  if (!P.early_writes) pdl_wait();
  for (int p = lo; p < hi; ++p) write_new_row<D, EB>(P, bi, j, p - p0, p, lane);
  return true;
}

// The tile count of every sequence as the CTAs see it: the exclusive prefix `cs` of the tile sums
// of nchunks chunks of `chunk` consecutive sequences (computed by each CTA in shared memory), and
// the lengths themselves for the tiles of one sequence.
struct TileIndex {
  const uint32_t* cs;   // [nchunks + 1]; cs[nchunks] = tiles of all sequences (per KV head)
  int chunk, nchunks;
  const int32_t* seq_lens;
  int B, g, n_max, T;
  __device__ __forceinline__ int tiles(int bi) const {
    return tiles_of_length(__ldg(seq_lens + bi), n_max, T);
  }
  // W: tiles of all segments
  __device__ __forceinline__ unsigned long long total() const {
    return static_cast<unsigned long long>(g) * cs[nchunks];
  }
};

// Walks the tiles of one CTA's range in segment order.
struct TileCursor {
  int bi, j, tile, nt;
  uint32_t pre;  // tiles of the sequences before bi (per KV head): segment (bi, j) starts at
                 // global tile g * pre + j * nt
  __device__ __forceinline__ void start(unsigned long long x, const TileIndex& ix) {
    const unsigned long long g = static_cast<unsigned long long>(ix.g);
    // the chunk holding tile x: the largest c with g * cs[c] <= x (it has tiles past x)
    int lo = 0, hi = ix.nchunks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g * ix.cs[mid] <= x) lo = mid; else hi = mid - 1;
    }
    uint32_t run = ix.cs[lo];
    int i = lo * ix.chunk;
    const int end = min(i + ix.chunk, ix.B);
    int t = 0;
    for (; i < end; ++i) {
      t = ix.tiles(i);
      if (g * (run + t) > x) break;
      run += t;
    }
    bi = min(i, ix.B - 1);
    pre = run;
    nt = max(ix.tiles(bi), 1);
    const unsigned long long rem = x - g * run;
    j = static_cast<int>(rem / nt);
    tile = static_cast<int>(rem % nt);
  }
  __device__ __forceinline__ void advance(const TileIndex& ix) {
    if (++tile < nt) return;
    tile = 0;
    if (++j < ix.g) return;
    j = 0;
    pre += nt;
    do {
      ++bi;
      nt = bi < ix.B ? ix.tiles(bi) : 0;
    } while (bi < ix.B && nt == 0);
  }
};

struct SharedLayout {
  uint8_t* stages;      // Geometry::kStages x kStageBytes, 1024-aligned
  float* comb_o;        // [NW][CR][comb_row_floats(D)]
  float2* comb_ml;      // [NW][CR]
  uint64_t* full;       // [stages]
  uint64_t* empty;      // [stages]
  uint64_t* cbar;       // consumer-wide barrier
  uint64_t* stall;      // testing: a barrier nothing completes (DecodeParams::debug_stall)
  volatile int* abort;  // set when any warp gives up
  volatile int* merge;  // this CTA is the last to arrive at the segment being finished
  int* pages;           // [2][32] paged caches: the pages of the tiles being issued (per producer)
  float* q_f32;         // the segment's q in fp32 (CcConsumer2), laid out by cc_q_index
  float* p_cc;          // [NW][kMaxCcHeads][kCcWarpKeys] key weights of a tile (CcConsumer2)
  TileIndex tix;        // tiles per sequence (its cs lives in static shared memory)
};

template <int D, int EB, int NW, int CR, int RB = kRingBytes>
__device__ __forceinline__ SharedLayout carve_shared(uint8_t* raw) {
  using Geo = Geometry<D, EB, RB>;
  constexpr int kStages = Geo::kStages;
  static_assert((NW * CR * comb_row_floats(D) * 4) % 16 == 0 && (NW * CR * 8) % 16 == 0 &&
                    ((2 * kStages + 2) * 8) % 16 == 0,
                "regions keep 16-byte alignment (the page slots are read as int4)");
  SharedLayout s;
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  s.stages = p;
  p += kStages * Geo::kStageBytes;
  s.comb_o = reinterpret_cast<float*>(p);
  p += NW * CR * comb_row_floats(D) * 4;
  s.comb_ml = reinterpret_cast<float2*>(p);
  p += NW * CR * 8;
  s.full = reinterpret_cast<uint64_t*>(p);
  s.empty = s.full + kStages;
  s.cbar = s.empty + kStages;
  s.stall = s.cbar + 1;
  p += (2 * kStages + 2) * 8;
  s.abort = reinterpret_cast<volatile int*>(p);
  s.merge = s.abort + 1;
  p += 16;
  s.pages = reinterpret_cast<int*>(p);  // 16-byte aligned: every region before it is a multiple
  p += kPagedProducers * 32 * 4;         // of 16 bytes
  s.q_f32 = reinterpret_cast<float*>(p);
  p += kMaxCcHeads * cc_q_row_floats(D) * 4;
  s.p_cc = reinterpret_cast<float*>(p);
  p += NW * kMaxCcHeads * kCcWarpKeys * 4;
  return s;
}

// Consumer-wide barrier on an mbarrier (all 32 * NW consumer threads arrive), bounded in time.
__device__ __forceinline__ bool consumer_sync(const SharedLayout& sh, uint32_t& phase,
                                              unsigned long long limit) {
  mbar_arrive(sh.cbar);
  const bool ok = mbar_wait_bounded(sh.cbar, phase, limit, sh.abort);
  phase ^= 1u;
  return ok;
}

// A wait of this thread ran out of time at `site` (tile k of the CTA's range): record where,
// latch MQA_ERR_TIMEOUT and tell the CTA's other warps to stop.
__device__ __forceinline__ void give_up(const SharedLayout& sh, int site, int k) {
  record_timeout_site(site, k);
  latch_status(kStatusTimeout);
  *sh.abort = 1;
}

// ---------------------------------------------------------------------------------------------
// Combine the consumer warps' states for one segment and write the result: the final bf16 output
// when the whole segment lies in this CTA, else a partial state in workspace slot `slot`.
// Row `hr` (a head of the group) has contributions at comb[(w, r)] for the pairs rows_of() gives.
// ---------------------------------------------------------------------------------------------
template <int D, int NW, int CR, class RowMap>
__device__ __forceinline__ void combine_and_store(const DecodeParams& P, const SharedLayout& sh,
                                                  int bi, int j, bool complete, int slot,
                                                  RowMap rows_of) {
  const int tid = threadIdx.x;  // 0 .. 32 * NW - 1 (consumer threads)
  const int G = P.G;
  for (int idx = tid; idx < G * D; idx += NW * 32) {
    const int hr = idx / D;
    const int d = idx - hr * D;
    int ws[NW], rs[NW];
    const int n = rows_of(hr, ws, rs);
    float M = -INFINITY;
    for (int c = 0; c < n; ++c) M = fmaxf(M, sh.comb_ml[ws[c] * CR + rs[c]].x);
    float acc = 0.f, den = 0.f;
    for (int c = 0; c < n; ++c) {
      const float2 ml = sh.comb_ml[ws[c] * CR + rs[c]];
      // a row that saw no key in this piece (an earlier token, T > 1) adds nothing
      const float wgt = (M == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
      den += wgt * ml.y;
      acc += wgt * sh.comb_o[(ws[c] * CR + rs[c]) * comb_row_floats(D) + d];
    }
    if (complete) {
      const size_t o = row_offset(P, bi, j, hr, D) + d;
      P.out[o] = __float2bfloat16_rn(acc / den * P.out_scale);
    } else {
      const size_t r = static_cast<size_t>(slot) * G + hr;
      P.part_o[r * D + d] = acc;
      if (d == 0) P.part_ml[r] = make_float2(M, den);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// The CTAs whose tile ranges cover a segment's tiles [s0, s1]: c_first .. c_last, skipping CTAs
// whose range is empty (only possible when W < P). CTA owning tile x: the largest c with
// c*W/P <= x, i.e. ((x+1)*P - 1) / W.
// ---------------------------------------------------------------------------------------------
struct SegmentPieces {
  int c_first, c_last;
  bool all_own;            // W >= P: every CTA owns at least one tile
  unsigned long long W, Pn;
  __device__ __forceinline__ SegmentPieces(unsigned long long s0, unsigned long long s1,
                                           unsigned long long W_, int P_)
      : W(W_), Pn(static_cast<unsigned long long>(P_)) {
    c_first = static_cast<int>(((s0 + 1) * Pn - 1) / W);
    c_last = static_cast<int>(((s1 + 1) * Pn - 1) / W);
    all_own = W >= Pn;
  }
  __device__ __forceinline__ bool owns(int c) const {
    return all_own || (W * static_cast<unsigned long long>(c) / Pn <
                       W * static_cast<unsigned long long>(c + 1) / Pn);
  }
  __device__ __forceinline__ unsigned int count() const {
    if (all_own) return static_cast<unsigned int>(c_last - c_first + 1);
    unsigned int n = 0;
    for (int c = c_first; c <= c_last; ++c) n += owns(c) ? 1u : 0u;
    return n;
  }
};

// Merge the partial states of a segment split across CTAs (run by the 128 consumer threads of
// the last CTA to arrive):  M = max_c m_c,  o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.
// Partials written by other SMs are read from L2 (ld.global.cg), never from a stale L1 line.
//
// This usually runs at the very end of the kernel (the CTA whose range ends inside a long segment
// arrives last), so it is written for latency: the pieces' (m, l) are staged in shared memory with
// independent loads, the per-head weights 2^(m_c - M) / l are computed once, and each output
// element then issues the loads of all pieces at once. Returns false if a barrier timed out.
template <int D, int NW, int CR>
__device__ __forceinline__ bool merge_split_segment(const DecodeParams& P, const SharedLayout& sh,
                                                    uint32_t& cphase, int bi, int j, int seg,
                                                    const SegmentPieces& pc) {
  const int G = P.G;
  const int tid = threadIdx.x;
  const int np = pc.c_last - pc.c_first + 1;
  constexpr int kScratchFloats = NW * CR * comb_row_floats(D);
  if (!pc.all_own || 3 * np * G > kScratchFloats) {
    // general case (some CTAs own no tiles, or too many pieces to stage): plain loops
    for (int idx = tid; idx < G * D; idx += NW * 32) {
      const int hr = idx / D;
      const int d = idx - hr * D;
      float M = -INFINITY;
      for (int c = pc.c_first; c <= pc.c_last; ++c)
        if (pc.owns(c)) M = fmaxf(M, __ldcg(P.part_ml + static_cast<size_t>(c + seg) * G + hr).x);
      float acc = 0.f, den = 0.f;
      for (int c = pc.c_first; c <= pc.c_last; ++c) {
        if (!pc.owns(c)) continue;
        const size_t r = static_cast<size_t>(c + seg) * G + hr;
        const float2 ml = __ldcg(P.part_ml + r);
        const float w = fast_exp2(ml.x - M);
        den += w * ml.y;
        acc += w * __ldcg(P.part_o + r * D + d);
      }
      P.out[row_offset(P, bi, j, hr, D) + d] = __float2bfloat16_rn(acc / den * P.out_scale);
    }
    return true;
  }
  // the combine scratch is free here: stage (m, l) of every piece, then the weights
  float2* ml = reinterpret_cast<float2*>(sh.comb_o);  // [np][G]
  float* wgt = sh.comb_o + 2 * np * G;                  // [np][G]
  const size_t slot0 = static_cast<size_t>(pc.c_first + seg);
  for (int e = tid; e < np * G; e += NW * 32) ml[e] = __ldcg(P.part_ml + slot0 * G + e);
  if (!consumer_sync(sh, cphase, P.timeout_ns)) return false;
  for (int hr = tid; hr < G; hr += NW * 32) {
    float M = -INFINITY;
    for (int pi = 0; pi < np; ++pi) M = fmaxf(M, ml[pi * G + hr].x);
    float den = 0.f;
    for (int pi = 0; pi < np; ++pi) den += fast_exp2(ml[pi * G + hr].x - M) * ml[pi * G + hr].y;
    const float inv = 1.f / den;
    for (int pi = 0; pi < np; ++pi) wgt[pi * G + hr] = fast_exp2(ml[pi * G + hr].x - M) * inv;
  }
  if (!consumer_sync(sh, cphase, P.timeout_ns)) return false;
  // outputs, four consecutive columns per thread
  const float4* po = reinterpret_cast<const float4*>(P.part_o);
  for (int idx = tid; idx < G * D / 4; idx += NW * 32) {
    const int hr = idx / (D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int pi = 0; pi < np; ++pi) {
      const float w = wgt[pi * G + hr];
      const float4 o = __ldcg(po + (slot0 + pi) * G * (D / 4) + idx);
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(
        P.out + row_offset(P, bi, j, hr, D) + (idx - hr * (D / 4)) * 4);
    const float os = P.out_scale;
    dst[0] = __floats2bfloat162_rn(acc.x * os, acc.y * os);
    dst[1] = __floats2bfloat162_rn(acc.z * os, acc.w * os);
  }
  // the scratch is written again by the next segment's combine
  return consumer_sync(sh, cphase, P.timeout_ns);
}

// ---------------------------------------------------------------------------------------------
// After this CTA stored its partial state of segment (bi, j) (and fenced it, and the consumer
// threads synchronised): count the arrival, and if this CTA is the last of the segment's pieces,
// merge them into the output and reset the counter. Run by the 32 * NW consumer threads; returns
// false if a barrier timed out.
// ---------------------------------------------------------------------------------------------
template <int D, int NW, int CR>
__device__ __forceinline__ bool finish_split_segment(const DecodeParams& P, const SharedLayout& sh,
                                                     uint32_t& cphase, const TileCursor& cur,
                                                     unsigned long long W) {
  const int bi = cur.bi, j = cur.j, nt = cur.nt;
  const int seg = bi * P.g + j;
  const unsigned long long s0 = static_cast<unsigned long long>(P.g) * cur.pre +
                                static_cast<unsigned long long>(j) * nt;
  const SegmentPieces pc(s0, s0 + nt - 1, W, P.num_ctas);
  if (threadIdx.x == 0) {
    // The partial rows were stored by many threads, ordered before this point by their fences and
    // the consumer barrier (CTA scope). The counter is the only thing other CTAs observe, so this
    // thread's fence before the increment is what releases those rows at device scope, and its
    // fence after it acquires the other pieces' rows before this CTA may merge them.
    __threadfence();
    const unsigned int before = atomicAdd(P.seg_arrivals + seg, 1u);
    __threadfence();
    *sh.merge = (before + 1u == pc.count()) ? 1 : 0;
  }
  if (!consumer_sync(sh, cphase, P.timeout_ns)) return false;
  if (P.debug_stall == 2 && !mbar_wait_bounded(sh.stall, 0, P.timeout_ns, sh.abort)) {
    // testing: give up with this arrival counted and no merge done, leaving the counter dirty
    if (!*sh.abort) give_up(sh, kSiteStall, 0);
    return false;
  }
  if (*sh.merge) {
    __threadfence();
    if (!merge_split_segment<D, NW, CR>(P, sh, cphase, bi, j, seg, pc)) return false;
    if (threadIdx.x == 0) P.seg_arrivals[seg] = 0u;  // ready for the next call
  }
  return true;
}

// ---------------------------------------------------------------------------------------------
// Prologue shared by the kernels: thread t sums the tiles of sequences [t * chunk, (t+1) * chunk)
// and the sums are scanned into sh.tix.cs[0 .. kThreads] (shared memory the caller provides), so
// that every CTA knows W and can find its tiles. Ends with a CTA-wide barrier, which also
// publishes barrier initialisation done before the call.
// ---------------------------------------------------------------------------------------------
template <int kThreads>
__device__ __forceinline__ void build_tile_prefix(const DecodeParams& P, SharedLayout& sh,
                                                  uint32_t* cs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = P.b;
  const int chunk = (B + kThreads - 1) / kThreads;
  const int lo = min(tid * chunk, B), hi = min(lo + chunk, B);
  uint32_t s = 0;
  for (int i = lo; i < hi; ++i) s += tiles_of_length(__ldg(P.seq_lens + i), P.n_max, P.T);
  cs[tid] = s;
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the kThreads chunk sums: each lane takes kPer consecutive ones, the lanes'
    // totals are scanned with shuffles
    constexpr int kPer = kThreads / 32;
    static_assert(kThreads % 32 == 0, "whole warps");
    uint32_t loc[kPer], tot = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) { loc[i] = cs[lane * kPer + i]; tot += loc[i]; }
    uint32_t incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    uint32_t run = incl - tot;
#pragma unroll
    for (int i = 0; i < kPer; ++i) { cs[lane * kPer + i] = run; run += loc[i]; }
    if (lane == 31) cs[kThreads] = incl;
  }
  __syncthreads();
  sh.tix.cs = cs;
  sh.tix.chunk = max(chunk, 1);
  sh.tix.nchunks = kThreads;
  sh.tix.seq_lens = P.seq_lens;
  sh.tix.B = B;
  sh.tix.g = P.g;
  sh.tix.n_max = P.n_max;
  sh.tix.T = P.T;
}

// Sequences whose length is out of range get a zero output and latch MQA_ERR_DEVICE_BOUNDS.
template <int D>
__device__ __forceinline__ void zero_invalid_sequences(const DecodeParams& P, int nthreads) {
  for (int bi = blockIdx.x; bi < P.b; bi += P.num_ctas) {
    const int L = __ldg(P.seq_lens + bi);
    if (L >= P.T && L <= P.n_max) continue;
    if (threadIdx.x == 0) latch_status(kStatusDeviceBounds);
    if (!P.early_writes) pdl_wait();
    __nv_bfloat16* ob = P.out + static_cast<size_t>(bi) * P.T * P.h * D;
    for (int e = threadIdx.x; e < P.T * P.h * D; e += nthreads) ob[e] = __float2bfloat16_rn(0.f);
  }
}

// ---------------------------------------------------------------------------------------------
// Producer warps: stream the CTA's tiles [x0, x0 + ntiles) into the stage ring with bulk tensor
// copies (one elected lane per warp), after writing the fused append's new row into the cache
// when the tile holds it (whole warp, one 16-byte chunk per lane). With np producer warps, warp
// pi issues tiles pi, pi + np, ...; np divides the stage count, so every stage is refilled by one
// warp, once its `empty` barrier has completed the phase of its previous use.
// ---------------------------------------------------------------------------------------------
template <int D, int EB, int RB = kRingBytes>
__device__ __forceinline__ void produce_tiles(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                              const DecodeParams& P, const SharedLayout& sh,
                                              unsigned long long x0, int ntiles, int lane,
                                              int np, int pi) {
  using Geo = Geometry<D, EB, RB>;
  constexpr int kStages = Geo::kStages;
  constexpr uint32_t kStageBytes = Geo::kStageBytes;
  constexpr uint32_t kKvBytes = Geo::kKvBytes;
  const bool fused = P.pos != nullptr;
  if (lane == 0) {
    prefetch_tensor_map(tm_k);
    prefetch_tensor_map(tm_v);
  }
  const uint64_t policy = l2_policy_evict_first();
  const int nmine = ntiles > pi ? (ntiles - pi + np - 1) / np : 0;
  if (nmine == 0) return;
  TileCursor cur;
  cur.start(x0 + static_cast<unsigned long long>(pi), sh.tix);
  int issued = 0;
  int row_bi = -1, row_p = -1;  // the first append row of sequence row_bi (-1: none to write)
  for (int i = 0; i < nmine; ++i) {
    const int k = pi + i * np;
    const int st = k % kStages;
    const uint32_t par = ((k / kStages) & 1) ^ 1;
    // the whole warp waits (no branch on the lane); a vote keeps the outcome warp-uniform
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait_bounded(&sh.empty[st], par, P.timeout_ns, sh.abort));
    if (!ok) {
      if (lane == 0 && !*sh.abort) give_up(sh, kSiteProducerEmpty, k);
      break;
    }
    if (fused) {
      if (cur.bi != row_bi) {
        row_bi = cur.bi;
        const int p = __ldg(P.pos + cur.bi);
        row_p = (p >= 0 && static_cast<long long>(p) + P.T <= P.n_max) ? p : -1;
      }
      if (row_p >= 0 && write_tile_rows<D, EB>(P, cur.bi, cur.j, cur.tile, row_p, lane)) {
        fence_proxy_async_global();  // each writer orders its store before the async proxy...
        __syncwarp();                // ...and the copy is issued after every writer
      }
    }
    // every lane holds the same values here; one elected lane issues the tile's copies
    if (elect_one()) {
      mbar_arrive_expect_tx(&sh.full[st], kStageBytes);
      const int z = cur.bi * P.g + cur.j;
      const int y = cur.tile * kTileKeys;
      uint8_t* kdst = sh.stages + st * kStageBytes;
      uint8_t* vdst = kdst + kKvBytes;
#pragma unroll
      for (int half = 0; half < Geo::kHalves; ++half) {
        tma_load_3d(kdst + half * kTileKeys * kSwizzleRowBytes, tm_k, &sh.full[st],
                    half * Geo::kBoxCols, y, z, policy);
        tma_load_3d(vdst + half * kTileKeys * kSwizzleRowBytes, tm_v, &sh.full[st],
                    half * Geo::kBoxCols, y, z, policy);
      }
    }
    __syncwarp();
    ++issued;
    for (int a = 0; a < np; ++a) cur.advance(sh.tix);
  }
  if (lane != 0 || issued == 0) return;
  // let this warp's copies still in flight land before the CTA may exit (bounded; no-op
  // normally): with np dividing the stage count, the tiles within kStages of its last one
  const volatile int never = 0;
  const int k_last = pi + (issued - 1) * np;
  for (int i = 0; i < issued; ++i) {
    const int k = pi + i * np;
    if (k > k_last - kStages)
      mbar_wait_bounded(&sh.full[k % kStages], (k / kStages) & 1, P.drain_ns, &never);
  }
}

// ---------------------------------------------------------------------------------------------
// Producer warp over paged caches. The tensor maps view each pool as (D, page_size,
// num_pages * g) with boxes of R = min(page_size, kTileKeys) rows, so a tile's rows
// [y, y + kTileKeys) arrive as up to NB = kTileKeys / R boxes: box i holds rows
// y + i R .. y + (i+1) R - 1, found at row (y + i R) % page_size of page
// page_table[bi][(y + i R) / page_size]. Every box lands at a multiple of R * 128 bytes (>= 1 KB)
// inside the stage, so the 128-byte swizzle comes out exactly as one box of the whole tile would
// give it. Boxes wholly at or past the length are not loaded (those stage rows are never used). A
// page index out of range latches MQA_ERR_DEVICE_BOUNDS and its box is read at a coordinate past
// the pool, which the copy fills with zeros, so the sequence attends over zero rows there.
//
// The producer is a single warp whose issue rate bounds the whole CTA once a tile takes several
// copies, so its per-tile path is kept short: page sizes are powers of two (shifts and masks, no
// division), NB is a compile-time constant, and the page-table reads are taken off the path. The
// warp looks up the pages of T = 32 / NB tiles at once (lane l: box l % NB of tile l / NB of the
// batch), one batch ahead of the tiles being issued, so each lookup's latency overlaps the batch
// before it; at a batch's start the lanes leave its pages in 32 shared-memory slots, from which
// one elected lane reads each tile's pages while it issues the tile's copies in one pass. A lookup reads only table entries below max_pages,
// possibly some past the sequence's length, whose values are never used.
// ---------------------------------------------------------------------------------------------
// Cursor of tile `base position + delta` of the CTA's range (global tile index x): the same
// segment as `base` when it still has that many tiles, else a fresh search.
__device__ __forceinline__ TileCursor cursor_ahead(const TileCursor& base, int delta,
                                                   unsigned long long x, const TileIndex& ix) {
  TileCursor c = base;
  if (base.tile + delta < base.nt) c.tile = base.tile + delta;
  else c.start(x, ix);
  return c;
}

// The page holding box `lane % NB` of the tile at `c` (0 where that box starts past n_max).
template <int NB>
__device__ __forceinline__ int lookup_page(const DecodeParams& P, const TileCursor& c, int lane,
                                           int page_shift) {
  constexpr int R = kTileKeys / NB;
  const int r = c.tile * kTileKeys + (lane % NB) * R;
  if (r >= P.n_max) return 0;
  return __ldg(P.page_table + static_cast<size_t>(c.bi) * P.max_pages + (r >> page_shift));
}

// The NB pages of tile kt of the current batch from the shared slots (16-byte aligned), with
// vector loads.
template <int NB>
__device__ __forceinline__ void load_tile_pages(const int* slots, int kt, int (&pg)[NB]) {
  if constexpr (NB == 8) {
    const int4 a = reinterpret_cast<const int4*>(slots)[2 * kt];
    const int4 b = reinterpret_cast<const int4*>(slots)[2 * kt + 1];
    pg[0] = a.x; pg[1] = a.y; pg[2] = a.z; pg[3] = a.w;
    pg[4] = b.x; pg[5] = b.y; pg[6] = b.z; pg[7] = b.w;
  } else if constexpr (NB == 4) {
    const int4 a = reinterpret_cast<const int4*>(slots)[kt];
    pg[0] = a.x; pg[1] = a.y; pg[2] = a.z; pg[3] = a.w;
  } else if constexpr (NB == 2) {
    const int2 a = reinterpret_cast<const int2*>(slots)[kt];
    pg[0] = a.x; pg[1] = a.y;
  } else {
    pg[0] = slots[kt];
  }
}

// Several producer warps share a CTA's tiles over paged caches (np of them; this one is number
// pi): warp pi issues tiles pi, pi + np, ... with its own page lookups and its own 32 slots.
template <int D, int EB, int NB, int RB = kRingBytes>
__device__ __forceinline__ void produce_tiles_paged(const CUtensorMap* tm_k,
                                                    const CUtensorMap* tm_v,
                                                    const DecodeParams& P, const SharedLayout& sh,
                                                    unsigned long long x0, int ntiles, int lane,
                                                    int np, int pi) {
  using Geo = Geometry<D, EB, RB>;
  constexpr int kStages = Geo::kStages;
  constexpr uint32_t kStageBytes = Geo::kStageBytes;
  constexpr uint32_t kKvBytes = Geo::kKvBytes;
  constexpr int R = kTileKeys / NB;  // rows per box
  constexpr int T = 32 / NB;         // tiles per lookup batch
  constexpr uint32_t kBoxBytes = R * kSwizzleRowBytes;
  const bool fused = P.pos != nullptr;
  const int page_shift = __ffs(P.page_size) - 1;
  const int page_mask = P.page_size - 1;
  const int z_past_pool = P.num_pages * P.g;
  if (lane == 0) {
    prefetch_tensor_map(tm_k);
    prefetch_tensor_map(tm_v);
  }
  const uint64_t policy = l2_policy_evict_first();
  const int my_tile = lane / NB;  // this lane's tile within a lookup batch
  int* slots = sh.pages + pi * 32;
  // this warp's tiles: k = pi + i * np for i < nmine
  const int nmine = ntiles > pi ? (ntiles - pi + np - 1) / np : 0;
  if (nmine == 0) return;
  TileCursor cur;
  cur.start(x0 + static_cast<unsigned long long>(pi), sh.tix);
  // `pages_next`: this lane's page of the next batch; `ahead`: the cursor of that batch's first tile
  TileCursor ahead = cur;
  int pages_next = 0;
  if (my_tile < nmine)
    pages_next = lookup_page<NB>(
        P, cursor_ahead(cur, my_tile * np, x0 + static_cast<unsigned long long>(pi + my_tile * np),
                        sh.tix),
        lane, page_shift);
  int issued = 0;
  int seq = -1, L = 0, row_p = -1;  // the sequence of the last tile, its length and append row
  for (int i = 0; i < nmine; ++i) {
    const int k = pi + i * np;
    const int kt = i % T;
    if (kt == 0) {
      // batch i / T starts: publish its pages (looked up a batch ago) to the slots and look up
      // the next batch
      __syncwarp();
      slots[lane] = pages_next;
      __syncwarp();
      const int i1 = i + T;
      if (i1 < nmine) {
        ahead = cursor_ahead(ahead, T * np, x0 + static_cast<unsigned long long>(pi + i1 * np),
                             sh.tix);
        if (i1 + my_tile < nmine)
          pages_next = lookup_page<NB>(
              P,
              cursor_ahead(ahead, my_tile * np,
                           x0 + static_cast<unsigned long long>(pi + (i1 + my_tile) * np), sh.tix),
              lane, page_shift);
      }
    }
    if (cur.bi != seq) {
      seq = cur.bi;
      L = __ldg(P.seq_lens + seq);
      if (fused) {
        const int p = __ldg(P.pos + seq);
        row_p = (p >= 0 && static_cast<long long>(p) + P.T <= P.n_max) ? p : -1;
      }
    }
    const int y = cur.tile * kTileKeys;
    const int st = k % kStages;
    const uint32_t par = ((k / kStages) & 1) ^ 1;
    // the whole warp waits (no branch on the lane); a vote keeps the outcome warp-uniform
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait_bounded(&sh.empty[st], par, P.timeout_ns, sh.abort));
    if (!ok) {
      if (lane == 0 && !*sh.abort) give_up(sh, kSiteProducerEmpty, k);
      break;
    }
    if (fused && row_p >= 0 && write_tile_rows<D, EB>(P, cur.bi, cur.j, cur.tile, row_p, lane)) {
      fence_proxy_async_global();
      __syncwarp();
    }
    // every lane holds the same values here; one elected lane issues the tile's copies
    if (elect_one()) {
      const int nbox = (min(L - y, kTileKeys) + R - 1) / R;  // L > y for every tile
      mbar_arrive_expect_tx(&sh.full[st],
                            static_cast<uint32_t>(nbox) * kBoxBytes * Geo::kHalves * 2);
      uint8_t* kdst = sh.stages + st * kStageBytes;
      uint8_t* vdst = kdst + kKvBytes;
      int pg[NB];
      load_tile_pages<NB>(slots, kt, pg);
      bool any_bad = false;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i < nbox) {
          const bool bad = static_cast<unsigned>(pg[i]) >= static_cast<unsigned>(P.num_pages);
          any_bad |= bad;
          const int z = bad ? z_past_pool : pg[i] * P.g + cur.j;
          const int yr = (y + i * R) & page_mask;
#pragma unroll
          for (int half = 0; half < Geo::kHalves; ++half) {
            tma_load_3d(kdst + half * kTileKeys * kSwizzleRowBytes + i * kBoxBytes, tm_k,
                        &sh.full[st], half * Geo::kBoxCols, yr, z, policy);
            tma_load_3d(vdst + half * kTileKeys * kSwizzleRowBytes + i * kBoxBytes, tm_v,
                        &sh.full[st], half * Geo::kBoxCols, yr, z, policy);
          }
        }
      }
      if (any_bad) latch_status(kStatusDeviceBounds);
    }
    __syncwarp();
    ++issued;
    for (int a = 0; a < np; ++a) cur.advance(sh.tix);
  }
  if (lane != 0 || issued == 0) return;
  // let this warp's copies still in flight land before the CTA may exit (bounded). With np
  // dividing the stage count, stage k % kStages only ever holds this warp's tiles, so a tile is
  // known to have landed once this warp has refilled its stage: the ones still to wait for are
  // those within kStages of the last tile it issued.
  const volatile int never = 0;
  const int k_last = pi + (issued - 1) * np;
  for (int i = 0; i < issued; ++i) {
    const int k = pi + i * np;
    if (k > k_last - kStages)
      mbar_wait_bounded(&sh.full[k % kStages], (k / kStages) & 1, P.drain_ns, &never);
  }
}

// Boxes per tile from the page size (8, 16, 32 rows; 64 or more: one box).
template <int D, int EB, int RB = kRingBytes>
__device__ __forceinline__ void produce_tiles_paged_any(const CUtensorMap* tm_k,
                                                        const CUtensorMap* tm_v,
                                                        const DecodeParams& P,
                                                        const SharedLayout& sh,
                                                        unsigned long long x0, int ntiles,
                                                        int lane, int np, int pi) {
  switch (P.page_size) {
    case 8: produce_tiles_paged<D, EB, 8, RB>(tm_k, tm_v, P, sh, x0, ntiles, lane, np, pi); break;
    case 16: produce_tiles_paged<D, EB, 4, RB>(tm_k, tm_v, P, sh, x0, ntiles, lane, np, pi); break;
    case 32: produce_tiles_paged<D, EB, 2, RB>(tm_k, tm_v, P, sh, x0, ntiles, lane, np, pi); break;
    default: produce_tiles_paged<D, EB, 1, RB>(tm_k, tm_v, P, sh, x0, ntiles, lane, np, pi); break;
  }
}

// ---------------------------------------------------------------------------------------------
// Tensor-core consumer (the automatic path from G = 3). WM warps (one per 16 heads) form a group; NW / WM groups split
// each tile's keys. kTokens: rows are (token, head) pairs of several new tokens, each masked by
// its own causal limit (instances used only when T > 1, so the single-token kernels carry no
// per-row state).
// ---------------------------------------------------------------------------------------------
template <int D, int WM, int NW, bool kTokens = false>
struct MmaConsumer {
  static constexpr int kWarps = NW;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = 1;
  static constexpr bool kSharedQ = false;
  static constexpr int kCombRows = 16;  // head rows per warp
  static constexpr int NGRP = NW / WM;
  static constexpr int KPW = kTileKeys / NGRP;  // keys per group per tile
  static constexpr int NT_S = KPW / 8;          // score tiles (n = 8 keys)
  static constexpr int KS_QK = D / 16;          // k-steps over the head dimension
  static constexpr int NT_O = D / 8;            // output tiles (n = 8 columns)
  static constexpr int KS_PV = KPW / 16;        // k-steps over keys
  static_assert(NT_S % 2 == 0 && KS_PV >= 1, "tile split");

  uint32_t qa[KS_QK][4];
  float o[NT_O][4];
  float ol[4];  // P 1: the running sums of the rounded weights, rescaled with O (all columns equal)
  float m[2];
  int lags;  // keys of a tile that rows r0 (low 16 bits) and r1 (high) do not see, relative to
             // the last token

  __device__ __forceinline__ void begin_segment(const DecodeParams& P, int bi, int j, int mi,
                                                int lane) {
    const int r0 = mi * 16 + (lane >> 2), r1 = r0 + 8;
    const bool v0 = r0 < P.G, v1 = r1 < P.G;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(P.q + (v0 ? row_offset(P, bi, j, r0, D) : 0));
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(P.q + (v1 ? row_offset(P, bi, j, r1, D) : 0));
    if constexpr (kTokens) lags = row_lag(P, r0) | (row_lag(P, r1) << 16);
#pragma unroll
    for (int ks = 0; ks < KS_QK; ++ks) {
      const int c = (ks * 16 + (lane & 3) * 2) >> 1;  // in bf16 pairs
      qa[ks][0] = v0 ? __ldg(q0 + c) : 0u;
      qa[ks][1] = v1 ? __ldg(q1 + c) : 0u;
      qa[ks][2] = v0 ? __ldg(q0 + c + 4) : 0u;
      qa[ks][3] = v1 ? __ldg(q1 + c + 4) : 0u;
    }
#pragma unroll
    for (int n = 0; n < NT_O; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    ol[0] = ol[1] = ol[2] = ol[3] = 0.f;
    m[0] = m[1] = -INFINITY;
  }

  // One tile. `valid` = rows of the sequence from this tile's first row on (at least 1; may
  // exceed the tile): key k of the tile is below the length when k < valid.
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int grp, int lane,
                                       int valid, float scale_log2) {
    // S = Q K^T, even and odd k-steps into separate accumulators (half the dependent chain)
    constexpr bool kSplit = true;
    float s[NT_S][4], s2[NT_S][4];
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.f;
    }
    const int mat = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int ks = 0; ks < KS_QK; ++ks) {
#pragma unroll
      for (int np = 0; np < NT_S / 2; ++np) {
        const int key = grp * KPW + np * 16 + rr + ((mat & 2) ? 8 : 0);
        const int d = ks * 16 + ((mat & 1) ? 8 : 0);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz(kbase, key, d), b0, b1, b2, b3);
        float (&acc0)[4] = (kSplit && (ks & 1)) ? s2[2 * np] : s[2 * np];
        float (&acc1)[4] = (kSplit && (ks & 1)) ? s2[2 * np + 1] : s[2 * np + 1];
        mma_16816(acc0, qa[ks], b0, b1);
        mma_16816(acc1, qa[ks], b2, b3);
      }
    }
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] += s2[n][0]; s[n][1] += s2[n][1]; s[n][2] += s2[n][2]; s[n][3] += s2[n][3];
    }
    // scale (log2 domain), mask keys a row does not see (at or past the length, or after the
    // row's token), running max per head row
    const int c2 = (lane & 3) * 2;
    const int va0 = kTokens ? valid - (lags & 0xFFFF) : valid;
    const int va1 = kTokens ? valid - (lags >> 16) : valid;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      const int key = grp * KPW + n * 8 + c2;
      s[n][0] = key < va0 ? s[n][0] * scale_log2 : -INFINITY;
      s[n][1] = key + 1 < va0 ? s[n][1] * scale_log2 : -INFINITY;
      s[n][2] = key < va1 ? s[n][2] * scale_log2 : -INFINITY;
      s[n][3] = key + 1 < va1 ? s[n][3] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
      mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // lazy reference: a row's reference m is raised (and its O and l rescaled) only when the
    // tile's maximum exceeds it by more than kLazyLog2, so most tiles leave O untouched and the
    // weights stay below 2^kLazyLog2. A row with no valid key yet keeps m = -inf.
    const bool up0 = mx0 > m[0] + kLazyLog2, up1 = mx1 > m[1] + kLazyLog2;
    float al0 = 1.f, al1 = 1.f;
    if (up0) { al0 = fast_exp2(m[0] - mx0); m[0] = mx0; }  // 0 when m was -inf
    if (up1) { al1 = fast_exp2(m[1] - mx1); m[1] = mx1; }
    const float ref0 = (m[0] == -INFINITY) ? 0.f : m[0];
    const float ref1 = (m[1] == -INFINITY) ? 0.f : m[1];
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] = fast_exp2(s[n][0] - ref0);
      s[n][1] = fast_exp2(s[n][1] - ref0);
      s[n][2] = fast_exp2(s[n][2] - ref1);
      s[n][3] = fast_exp2(s[n][3] - ref1);
    }
    if (__any_sync(0xffffffffu, up0 || up1)) {
#pragma unroll
      for (int n = 0; n < NT_O; ++n) {
        o[n][0] *= al0; o[n][1] *= al0;
        o[n][2] *= al1; o[n][3] *= al1;
      }
      ol[0] *= al0; ol[1] *= al0; ol[2] *= al1; ol[3] *= al1;
    }
    // O += P V with the weights rounded to bf16 once; P 1 on the tensor cores sums exactly those
    // rounded weights (fp32), so the normalised weights still add up to one
#pragma unroll
    for (int kk = 0; kk < KS_PV; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      mma_16816(ol, a, kOnesBf16x2, kOnesBf16x2);
#pragma unroll
      for (int dp = 0; dp < NT_O / 2; ++dp) {
        const int key = grp * KPW + kk * 16 + rr + ((mat & 1) ? 8 : 0);
        const int d = dp * 16 + ((mat & 2) ? 8 : 0);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(swz(vbase, key, d), b0, b1, b2, b3);
        mma_16816(o[2 * dp], a, b0, b1);
        mma_16816(o[2 * dp + 1], a, b2, b3);
      }
    }
  }

  // Publish this warp's state (rows mi*16 .. mi*16+15 of the group) to the combine scratch.
  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
    const float l0 = ol[0], l1 = ol[2];  // row sums over all of this warp's keys
    const int r = lane >> 2, c2 = (lane & 3) * 2;
    float* row0 = sh.comb_o + (warp * kCombRows + r) * comb_row_floats(D);
    float* row1 = sh.comb_o + (warp * kCombRows + r + 8) * comb_row_floats(D);
#pragma unroll
    for (int n = 0; n < NT_O; ++n) {
      *reinterpret_cast<float2*>(row0 + n * 8 + c2) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(row1 + n * 8 + c2) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      sh.comb_ml[warp * kCombRows + r] = make_float2(m[0], l0);
      sh.comb_ml[warp * kCombRows + r + 8] = make_float2(m[1], l1);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int grp = 0; grp < NGRP; ++grp) {
        ws[grp] = grp * WM + (hr >> 4);
        rs[grp] = hr & 15;
      }
      return NGRP;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// Tensor-core consumer for fp8 E4M3 caches (from G = 3): the same tile split, softmax and combine as
// MmaConsumer, with fp16 MMAs (m16n8k16, fp32 accumulate). The codes are widened exactly to fp16
// in registers (two codes per instruction); q is rounded to fp16 once per segment; the weights P
// are rounded to fp16 once, and the running sum takes the same rounded values. The per-tensor
// scales never enter here: k_scale is part of scale_log2 and v_scale multiplies the final output.
//
// S = Q K^T: ldmatrix reads the K stage as 16-bit units, so a lane receives four consecutive
// codes of one key (columns 4c .. 4c+3 of a 16-column block, c = lane % 4); widened, they are one
// whole B fragment of a k16 step whose k order is the permutation 2c, 2c+1 -> 4c, 4c+1 and
// 2c+8, 2c+9 -> 4c+2, 4c+3 of the block's columns. The A fragments of q use the same order, and
// a dot product does not depend on the order of its terms.
// O += P V: ldmatrix.trans on the V stage gives a lane two keys (rows 2c, 2c+1 of an 8-key block)
// times two adjacent columns (2r, 2r+1, r = lane / 4) of a 16-column block; one byte permute and
// two widenings give the B fragments of two n8 tiles, the block's even columns and its odd
// columns. Output tile 2b + e (block b, e = 0 even, 1 odd) thus holds columns 16b + 2n + e, and
// a lane's accumulators cover columns 16b + 4c + {0, 1, 2, 3}, which publish() writes back in
// order.
// Tile groups (TG = 2): an fp8 tile carries half the bytes of a bf16 one, so its HBM time is half
// while a warp's per-tile chain of dependent steps (ldmatrix, widening, MMAs, softmax, MMAs) is
// not shorter. Eight warps then form two groups of four that take alternate tiles of the CTA's
// range, each with its own softmax state, merged with the key groups at the segment's end; every
// warp still does a whole tile's worth of work per tile it owns.
// ---------------------------------------------------------------------------------------------
template <int D, int WM, int NW, int TG = 1>
struct MmaConsumerF8 {
  static constexpr int kWarps = NW;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = TG;
  static constexpr bool kSharedQ = false;
  static constexpr int kCombRows = 16;  // head rows per warp
  static constexpr int NGRP = NW / (WM * TG);  // key groups per tile group
  static constexpr int KPW = kTileKeys / NGRP;  // keys per group per tile
  static constexpr int NT_S = KPW / 8;          // score tiles (n = 8 keys)
  static constexpr int KS_QK = D / 16;          // k-steps over the head dimension
  static constexpr int NT_O = D / 8;            // output tiles (n = 8 columns)
  static constexpr int KS_PV = KPW / 16;        // k-steps over keys
  static_assert(D == 128 && NT_S % 2 == 0 && KS_PV >= 1 && KS_QK % 2 == 0, "tile split");

  uint32_t qa[KS_QK][4];
  float o[NT_O][4];
  float ol[4];  // P 1: the running sums of the rounded weights, rescaled with O (all columns equal)
  float m[2];

  __device__ __forceinline__ void begin_segment(const DecodeParams& P, int bi, int j, int mi,
                                                int lane) {
    const int r0 = mi * 16 + (lane >> 2), r1 = r0 + 8;
    const bool v0 = r0 < P.G, v1 = r1 < P.G;
    const uint2* q0 = reinterpret_cast<const uint2*>(P.q + (v0 ? row_offset(P, bi, j, r0, D) : 0));
    const uint2* q1 = reinterpret_cast<const uint2*>(P.q + (v1 ? row_offset(P, bi, j, r1, D) : 0));
#pragma unroll
    for (int ks = 0; ks < KS_QK; ++ks) {
      // columns 16 ks + 4c .. + 3 of rows r0 and r1 (one 8-byte load each)
      const int c4 = ks * 4 + (lane & 3);
      const uint2 x0 = v0 ? __ldg(q0 + c4) : make_uint2(0u, 0u);
      const uint2 x1 = v1 ? __ldg(q1 + c4) : make_uint2(0u, 0u);
      const __nv_bfloat162 a0 = *reinterpret_cast<const __nv_bfloat162*>(&x0.x);
      const __nv_bfloat162 a1 = *reinterpret_cast<const __nv_bfloat162*>(&x0.y);
      const __nv_bfloat162 b0 = *reinterpret_cast<const __nv_bfloat162*>(&x1.x);
      const __nv_bfloat162 b1 = *reinterpret_cast<const __nv_bfloat162*>(&x1.y);
      qa[ks][0] = pack_f16x2(__low2float(a0), __high2float(a0));
      qa[ks][1] = pack_f16x2(__low2float(b0), __high2float(b0));
      qa[ks][2] = pack_f16x2(__low2float(a1), __high2float(a1));
      qa[ks][3] = pack_f16x2(__low2float(b1), __high2float(b1));
    }
#pragma unroll
    for (int n = 0; n < NT_O; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    ol[0] = ol[1] = ol[2] = ol[3] = 0.f;
    m[0] = m[1] = -INFINITY;
  }

  // One tile. `valid` = rows of the sequence from this tile's first row on (at least 1; may
  // exceed the tile): key k of the tile is below the length when k < valid.
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int grp, int lane,
                                       int valid, float scale_log2) {
    // S = Q K^T, block ks into s and block ks + 1 into s2 (half the dependent chain)
    float s[NT_S][4], s2[NT_S][4];
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.f;
    }
    const int mat = lane >> 3, rr = lane & 7;
    // one ldmatrix.x4 = keys (8 or 8 + 8) x column blocks (ks, ks + 1)
#pragma unroll
    for (int ks = 0; ks < KS_QK; ks += 2) {
#pragma unroll
      for (int np = 0; np < NT_S / 2; ++np) {
        const int key = grp * KPW + np * 16 + rr + ((mat & 2) ? 8 : 0);
        uint32_t w0, w1, w2, w3;
        ldsm_x4(swz_bytes(kbase, key, (ks + (mat & 1)) * 16), w0, w1, w2, w3);
        uint32_t b[4][2];
        e4m3x4_to_f16x2x2(w0, b[0][0], b[0][1]);  // keys 0-7,  block ks
        e4m3x4_to_f16x2x2(w1, b[1][0], b[1][1]);  // keys 0-7,  block ks + 1
        e4m3x4_to_f16x2x2(w2, b[2][0], b[2][1]);  // keys 8-15, block ks
        e4m3x4_to_f16x2x2(w3, b[3][0], b[3][1]);  // keys 8-15, block ks + 1
        mma_16816_f16(s[2 * np], qa[ks], b[0][0], b[0][1]);
        mma_16816_f16(s2[2 * np], qa[ks + 1], b[1][0], b[1][1]);
        mma_16816_f16(s[2 * np + 1], qa[ks], b[2][0], b[2][1]);
        mma_16816_f16(s2[2 * np + 1], qa[ks + 1], b[3][0], b[3][1]);
      }
    }
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] += s2[n][0]; s[n][1] += s2[n][1]; s[n][2] += s2[n][2]; s[n][3] += s2[n][3];
    }
    // scale (log2 domain), mask rows at or beyond the length, running max per head row
    const int c2 = (lane & 3) * 2;
    const int va0 = valid, va1 = valid;  // one token: every row sees the same keys
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      const int key = grp * KPW + n * 8 + c2;
      s[n][0] = key < va0 ? s[n][0] * scale_log2 : -INFINITY;
      s[n][1] = key + 1 < va0 ? s[n][1] * scale_log2 : -INFINITY;
      s[n][2] = key < va1 ? s[n][2] * scale_log2 : -INFINITY;
      s[n][3] = key + 1 < va1 ? s[n][3] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
      mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // lazy reference, as in MmaConsumer::tile (weights stay below 2^kLazyLog2, well inside fp16)
    const bool up0 = mx0 > m[0] + kLazyLog2, up1 = mx1 > m[1] + kLazyLog2;
    float al0 = 1.f, al1 = 1.f;
    if (up0) { al0 = fast_exp2(m[0] - mx0); m[0] = mx0; }
    if (up1) { al1 = fast_exp2(m[1] - mx1); m[1] = mx1; }
    const float ref0 = (m[0] == -INFINITY) ? 0.f : m[0];
    const float ref1 = (m[1] == -INFINITY) ? 0.f : m[1];
#pragma unroll
    for (int n = 0; n < NT_S; ++n) {
      s[n][0] = fast_exp2(s[n][0] - ref0);
      s[n][1] = fast_exp2(s[n][1] - ref0);
      s[n][2] = fast_exp2(s[n][2] - ref1);
      s[n][3] = fast_exp2(s[n][3] - ref1);
    }
    if (__any_sync(0xffffffffu, up0 || up1)) {
#pragma unroll
      for (int n = 0; n < NT_O; ++n) {
        o[n][0] *= al0; o[n][1] *= al0;
        o[n][2] *= al1; o[n][3] *= al1;
      }
      ol[0] *= al0; ol[1] *= al0; ol[2] *= al1; ol[3] *= al1;
    }
    // O += P V with the weights rounded to fp16 once; P 1 sums exactly those rounded weights
#pragma unroll
    for (int kk = 0; kk < KS_PV; ++kk) {
      uint32_t a[4];
      a[0] = pack_f16x2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_f16x2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_f16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_f16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      mma_16816_f16(ol, a, kOnesF16x2, kOnesF16x2);
#pragma unroll
      for (int cb = 0; cb < D / 16; cb += 2) {
        // matrices: keys 0-7 / 8-15 of this k-step x column blocks cb / cb + 1
        const int key = grp * KPW + kk * 16 + rr + ((mat & 1) ? 8 : 0);
        uint32_t w0, w1, w2, w3;
        ldsm_x4_trans(swz_bytes(vbase, key, (cb + (mat >> 1)) * 16), w0, w1, w2, w3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // keys 0-7 and 8-15 of block cb + h: bytes (0, 2) are the even column, (1, 3) the odd
          uint32_t e0, o0, e1, o1;
          e4m3x4_to_f16x2x2(__byte_perm(h ? w2 : w0, 0u, 0x3120), e0, o0);
          e4m3x4_to_f16x2x2(__byte_perm(h ? w3 : w1, 0u, 0x3120), e1, o1);
          mma_16816_f16(o[2 * (cb + h)], a, e0, e1);
          mma_16816_f16(o[2 * (cb + h) + 1], a, o0, o1);
        }
      }
    }
  }

  // Publish this warp's state (rows mi*16 .. mi*16+15 of the group) to the combine scratch.
  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
    const float l0 = ol[0], l1 = ol[2];  // row sums over all of this warp's keys
    const int r = lane >> 2, c4 = (lane & 3) * 4;
    float* row0 = sh.comb_o + (warp * kCombRows + r) * comb_row_floats(D);
    float* row1 = sh.comb_o + (warp * kCombRows + r + 8) * comb_row_floats(D);
#pragma unroll
    for (int b = 0; b < D / 16; ++b) {
      // tiles 2b (even columns) and 2b + 1 (odd): columns 16b + 4c + {0, 2} and {1, 3}
      *reinterpret_cast<float4*>(row0 + b * 16 + c4) =
          make_float4(o[2 * b][0], o[2 * b + 1][0], o[2 * b][1], o[2 * b + 1][1]);
      *reinterpret_cast<float4*>(row1 + b * 16 + c4) =
          make_float4(o[2 * b][2], o[2 * b + 1][2], o[2 * b][3], o[2 * b + 1][3]);
    }
    if ((lane & 3) == 0) {
      sh.comb_ml[warp * kCombRows + r] = make_float2(m[0], l0);
      sh.comb_ml[warp * kCombRows + r + 8] = make_float2(m[1], l1);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int t = 0; t < TG; ++t) {
#pragma unroll
        for (int grp = 0; grp < NGRP; ++grp) {
          ws[t * NGRP + grp] = t * (NW / TG) + grp * WM + (hr >> 4);
          rs[t * NGRP + grp] = hr & 15;
        }
      }
      return TG * NGRP;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// Consumer over fp8 E4M3 caches for groups of at most 8 heads: the products of MmaConsumerF8,
// transposed. S^T = K q^T and O^T = V^T P^T put keys (then output columns) on the 16 rows of
// each m16n8k16 MMA and the group's heads on its 8 columns, so no MMA carries padding rows: half
// the MMAs, exponentials and accumulators of the head-row form, whose 16 rows hold 8 heads.
//
// S^T: one ldmatrix.x4 over the K stage gives a lane four consecutive codes (columns 4c .. 4c+3
// of a 16-column block, c = lane % 4) of key r and of key r + 8 (r = lane / 4) for two column
// blocks; widened, they are the A fragments of two k16 steps in the k order 2c, 2c+1 -> 4c, 4c+1
// and 2c+8, 2c+9 -> 4c+2, 4c+3, which the B fragments of q^T (head r of the group, zero past G)
// repeat.
// P^T: the accumulator of S^T holds keys r and r + 8 by heads 2c, 2c+1; rounded to fp16 and
// transposed with movmatrix it is the B fragment of P^T (head r by keys 2c, 2c+1 and 2c+8, 2c+9).
// O^T: ldmatrix.trans over the V stage gives a lane keys 2c, 2c+1 of columns 2r, 2r+1 of a
// 16-column block; one byte permute and two widenings make the A fragment whose rows r and r + 8
// are the block's columns 2r and 2r + 1. The accumulator of block b then holds columns 16b + 2r
// (c0, c1) and 16b + 2r + 1 (c2, c3) of heads 2c (c0, c2) and 2c + 1 (c1, c3).
// Tile groups and key groups as in MmaConsumerF8: the NW warps form TG groups that take turns on
// the tiles, and the NW / TG warps of a group split each tile's keys.
// ---------------------------------------------------------------------------------------------
template <int D, int NW, int TG>
struct MmaConsumerF8T {
  static constexpr int kWarps = NW;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = TG;
  static constexpr bool kSharedQ = false;
  static constexpr int kCombRows = 8;            // heads per warp
  static constexpr int NGRP = NW / TG;           // key groups per tile group
  static constexpr int KPW = kTileKeys / NGRP;   // keys per warp per tile
  static constexpr int MT_S = KPW / 16;          // m-tiles of S^T (16 keys each)
  static constexpr int KS_QK = D / 16;           // k-steps over the head dimension
  static constexpr int MT_O = D / 16;            // m-tiles of O^T (16 output columns each)
  static_assert(D == 128 && MT_S >= 1 && KS_QK % 2 == 0 && MT_O % 2 == 0, "tile split");

  uint32_t qb[KS_QK][2];  // B fragments of q^T for head lane / 4 of the group
  float o[MT_O][4];
  float ol[4];  // P^T summed over keys by an all-ones A: c0 head 2c, c1 head 2c + 1
  float m[2];   // softmax references of heads 2c and 2c + 1 (log2 units)

  __device__ __forceinline__ void begin_segment(const DecodeParams& P, int bi, int j, int mi,
                                                int lane) {
    const int r = lane >> 2;
    const bool valid = r < P.G;
    const uint2* qr = reinterpret_cast<const uint2*>(P.q + (valid ? row_offset(P, bi, j, r, D) : 0));
#pragma unroll
    for (int ks = 0; ks < KS_QK; ++ks) {
      // columns 16 ks + 4c .. + 3 of head r (one 8-byte load)
      const uint2 x = valid ? __ldg(qr + ks * 4 + (lane & 3)) : make_uint2(0u, 0u);
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x.x);
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x.y);
      qb[ks][0] = pack_f16x2(__low2float(a), __high2float(a));
      qb[ks][1] = pack_f16x2(__low2float(b), __high2float(b));
    }
#pragma unroll
    for (int n = 0; n < MT_O; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    ol[0] = ol[1] = ol[2] = ol[3] = 0.f;
    m[0] = m[1] = -INFINITY;
  }

  // One tile: this warp's KPW keys from grp * KPW. `valid` = rows of the sequence from the tile's
  // first row on (at least 1; may exceed the tile).
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int grp, int lane,
                                       int valid, float scale_log2) {
    const int mat = lane >> 3, rr = lane & 7;
    const int r = lane >> 2;
    // S^T, column blocks ks into s and ks + 1 into s2 (two independent chains per m-tile)
    float s[MT_S][4], s2[MT_S][4];
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
      s2[t][0] = s2[t][1] = s2[t][2] = s2[t][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < KS_QK; ks += 2) {
#pragma unroll
      for (int t = 0; t < MT_S; ++t) {
        // matrices: keys 0-7 / 8-15 of the m-tile x column blocks ks / ks + 1
        const int key = grp * KPW + t * 16 + rr + ((mat & 1) ? 8 : 0);
        uint32_t w0, w1, w2, w3;
        ldsm_x4(swz_bytes(kbase, key, (ks + (mat >> 1)) * 16), w0, w1, w2, w3);
        uint32_t a[4], a2[4];
        e4m3x4_to_f16x2x2(w0, a[0], a[2]);    // key r,     block ks
        e4m3x4_to_f16x2x2(w1, a[1], a[3]);    // key r + 8, block ks
        e4m3x4_to_f16x2x2(w2, a2[0], a2[2]);  // key r,     block ks + 1
        e4m3x4_to_f16x2x2(w3, a2[1], a2[3]);  // key r + 8, block ks + 1
        mma_16816_f16(s[t], a, qb[ks][0], qb[ks][1]);
        mma_16816_f16(s2[t], a2, qb[ks + 1][0], qb[ks + 1][1]);
      }
    }
    // scale (log2 domain), mask keys at or beyond the length, running max per head
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      const int key = grp * KPW + t * 16 + r;
      const bool in0 = key < valid, in1 = key + 8 < valid;
      s[t][0] = in0 ? (s[t][0] + s2[t][0]) * scale_log2 : -INFINITY;  // key r,     head 2c
      s[t][1] = in0 ? (s[t][1] + s2[t][1]) * scale_log2 : -INFINITY;  // key r,     head 2c + 1
      s[t][2] = in1 ? (s[t][2] + s2[t][2]) * scale_log2 : -INFINITY;  // key r + 8, head 2c
      s[t][3] = in1 ? (s[t][3] + s2[t][3]) * scale_log2 : -INFINITY;  // key r + 8, head 2c + 1
      mx0 = fmaxf(mx0, fmaxf(s[t][0], s[t][2]));
      mx1 = fmaxf(mx1, fmaxf(s[t][1], s[t][3]));
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // lazy reference, as in MmaConsumer::tile (weights stay below 2^kLazyLog2, well inside fp16)
    const bool up0 = mx0 > m[0] + kLazyLog2, up1 = mx1 > m[1] + kLazyLog2;
    float al0 = 1.f, al1 = 1.f;
    if (up0) { al0 = fast_exp2(m[0] - mx0); m[0] = mx0; }
    if (up1) { al1 = fast_exp2(m[1] - mx1); m[1] = mx1; }
    const float ref0 = (m[0] == -INFINITY) ? 0.f : m[0];
    const float ref1 = (m[1] == -INFINITY) ? 0.f : m[1];
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      s[t][0] = fast_exp2(s[t][0] - ref0);
      s[t][1] = fast_exp2(s[t][1] - ref1);
      s[t][2] = fast_exp2(s[t][2] - ref0);
      s[t][3] = fast_exp2(s[t][3] - ref1);
    }
    if (__any_sync(0xffffffffu, up0 || up1)) {
#pragma unroll
      for (int n = 0; n < MT_O; ++n) {
        o[n][0] *= al0; o[n][1] *= al1;
        o[n][2] *= al0; o[n][3] *= al1;
      }
      ol[0] *= al0; ol[1] *= al1; ol[2] *= al0; ol[3] *= al1;
    }
    // O^T += V^T P^T with the weights rounded to fp16 once; the all-ones A sums those weights
    const uint32_t ones[4] = {kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2};
#pragma unroll
    for (int kk = 0; kk < MT_S; ++kk) {
      const uint32_t b0 = movmatrix_trans(pack_f16x2(s[kk][0], s[kk][1]));  // keys 2c, 2c+1
      const uint32_t b1 = movmatrix_trans(pack_f16x2(s[kk][2], s[kk][3]));  // keys 2c+8, 2c+9
      mma_16816_f16(ol, ones, b0, b1);
#pragma unroll
      for (int cb = 0; cb < MT_O; cb += 2) {
        // matrices: keys 0-7 / 8-15 of this k-step x column blocks cb / cb + 1
        const int key = grp * KPW + kk * 16 + rr + ((mat & 1) ? 8 : 0);
        uint32_t w0, w1, w2, w3;
        ldsm_x4_trans(swz_bytes(vbase, key, (cb + (mat >> 1)) * 16), w0, w1, w2, w3);
        // bytes (0, 2) of a permuted word are column 2r of keys 2c, 2c+1; bytes (1, 3) column
        // 2r + 1
        uint32_t a[4], a2[4];
        e4m3x4_to_f16x2x2(__byte_perm(w0, 0u, 0x3120), a[0], a[1]);
        e4m3x4_to_f16x2x2(__byte_perm(w1, 0u, 0x3120), a[2], a[3]);
        e4m3x4_to_f16x2x2(__byte_perm(w2, 0u, 0x3120), a2[0], a2[1]);
        e4m3x4_to_f16x2x2(__byte_perm(w3, 0u, 0x3120), a2[2], a2[3]);
        mma_16816_f16(o[cb], a, b0, b1);
        mma_16816_f16(o[cb + 1], a2, b0, b1);
      }
    }
  }

  // Publish this warp's state (the group's heads 0..7) to the combine scratch.
  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
    const int r = lane >> 2, h0 = (lane & 3) * 2;
    float* row0 = sh.comb_o + (warp * kCombRows + h0) * comb_row_floats(D);
    float* row1 = row0 + comb_row_floats(D);
#pragma unroll
    for (int b = 0; b < MT_O; ++b) {
      *reinterpret_cast<float2*>(row0 + b * 16 + 2 * r) = make_float2(o[b][0], o[b][2]);
      *reinterpret_cast<float2*>(row1 + b * 16 + 2 * r) = make_float2(o[b][1], o[b][3]);
    }
    if (r == 0) {
      sh.comb_ml[warp * kCombRows + h0] = make_float2(m[0], ol[0]);
      sh.comb_ml[warp * kCombRows + h0 + 1] = make_float2(m[1], ol[1]);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        ws[w] = w;
        rs[w] = hr;
      }
      return NW;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// Consumer over bf16 caches for groups of at most 8 heads: the products transposed as in
// MmaConsumerF8T (S^T = K q^T, O^T = V^T P^T; keys, then output columns, on the 16 MMA rows and
// the group's heads on the 8 columns), with the tiles' bf16 rows taken by ldmatrix as they are.
// S^T: ldmatrix.x4 gives the A fragment of 16 keys by 16 columns directly; the B fragment of q^T
// is head r's columns (2c, 2c+1) and (2c+8, 2c+9) of the k-step, loaded once per segment.
// O^T: ldmatrix.x4.trans over the V stage gives the A fragment of 16 columns by 16 keys. P^T and
// the row sums as in MmaConsumerF8T. With four warps, each takes 16 keys of every tile.
// ---------------------------------------------------------------------------------------------
template <int D, int NW>
struct MmaConsumerT {
  static constexpr int kWarps = NW;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = 1;
  static constexpr bool kSharedQ = false;
  static constexpr int kCombRows = 8;            // heads per warp
  static constexpr int KPW = kTileKeys / NW;     // keys per warp per tile
  static constexpr int MT_S = KPW / 16;          // m-tiles of S^T (16 keys each)
  static constexpr int KS_QK = D / 16;           // k-steps over the head dimension
  static constexpr int MT_O = D / 16;            // m-tiles of O^T (16 output columns each)
  static_assert(MT_S >= 1 && KS_QK % 2 == 0, "tile split");

  uint32_t qb[KS_QK][2];  // B fragments of q^T for head lane / 4 of the group
  float o[MT_O][4];
  float ol[4];  // P^T summed over keys by an all-ones A: c0 head 2c, c1 head 2c + 1
  float m[2];   // softmax references of heads 2c and 2c + 1 (log2 units)

  __device__ __forceinline__ void begin_segment(const DecodeParams& P, int bi, int j, int mi,
                                                int lane) {
    const int r = lane >> 2, c = lane & 3;
    const bool valid = r < P.G;
    const uint32_t* qr =
        reinterpret_cast<const uint32_t*>(P.q + (valid ? row_offset(P, bi, j, r, D) : 0));
#pragma unroll
    for (int ks = 0; ks < KS_QK; ++ks) {
      // columns 16 ks + 2c, + 1 and 16 ks + 8 + 2c, + 1 of head r
      qb[ks][0] = valid ? __ldg(qr + ks * 8 + c) : 0u;
      qb[ks][1] = valid ? __ldg(qr + ks * 8 + 4 + c) : 0u;
    }
#pragma unroll
    for (int n = 0; n < MT_O; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    ol[0] = ol[1] = ol[2] = ol[3] = 0.f;
    m[0] = m[1] = -INFINITY;
  }

  // One tile: this warp's KPW keys from grp * KPW. `valid` = rows of the sequence from the tile's
  // first row on (at least 1; may exceed the tile).
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int grp, int lane,
                                       int valid, float scale_log2) {
    const int mat = lane >> 3, rr = lane & 7;
    const int r = lane >> 2;
    // S^T, k-steps ks into s and ks + 1 into s2 (two independent chains per m-tile)
    float s[MT_S][4], s2[MT_S][4];
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
      s2[t][0] = s2[t][1] = s2[t][2] = s2[t][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < KS_QK; ks += 2) {
#pragma unroll
      for (int t = 0; t < MT_S; ++t) {
        // matrices: keys 0-7 / 8-15 of the m-tile (mat & 1) x columns + 0-7 / + 8-15 (mat >> 1)
        const int key = grp * KPW + t * 16 + rr + ((mat & 1) ? 8 : 0);
        uint32_t a[4], a2[4];
        ldsm_x4(swz_bytes(kbase, key, ks * 32 + (mat >> 1) * 16), a[0], a[1], a[2], a[3]);
        ldsm_x4(swz_bytes(kbase, key, (ks + 1) * 32 + (mat >> 1) * 16), a2[0], a2[1], a2[2],
                a2[3]);
        mma_16816(s[t], a, qb[ks][0], qb[ks][1]);
        mma_16816(s2[t], a2, qb[ks + 1][0], qb[ks + 1][1]);
      }
    }
    // scale (log2 domain), mask keys at or beyond the length, running max per head
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      const int key = grp * KPW + t * 16 + r;
      const bool in0 = key < valid, in1 = key + 8 < valid;
      s[t][0] = in0 ? (s[t][0] + s2[t][0]) * scale_log2 : -INFINITY;  // key r,     head 2c
      s[t][1] = in0 ? (s[t][1] + s2[t][1]) * scale_log2 : -INFINITY;  // key r,     head 2c + 1
      s[t][2] = in1 ? (s[t][2] + s2[t][2]) * scale_log2 : -INFINITY;  // key r + 8, head 2c
      s[t][3] = in1 ? (s[t][3] + s2[t][3]) * scale_log2 : -INFINITY;  // key r + 8, head 2c + 1
      mx0 = fmaxf(mx0, fmaxf(s[t][0], s[t][2]));
      mx1 = fmaxf(mx1, fmaxf(s[t][1], s[t][3]));
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // lazy reference, as in MmaConsumer::tile
    const bool up0 = mx0 > m[0] + kLazyLog2, up1 = mx1 > m[1] + kLazyLog2;
    float al0 = 1.f, al1 = 1.f;
    if (up0) { al0 = fast_exp2(m[0] - mx0); m[0] = mx0; }
    if (up1) { al1 = fast_exp2(m[1] - mx1); m[1] = mx1; }
    const float ref0 = (m[0] == -INFINITY) ? 0.f : m[0];
    const float ref1 = (m[1] == -INFINITY) ? 0.f : m[1];
#pragma unroll
    for (int t = 0; t < MT_S; ++t) {
      s[t][0] = fast_exp2(s[t][0] - ref0);
      s[t][1] = fast_exp2(s[t][1] - ref1);
      s[t][2] = fast_exp2(s[t][2] - ref0);
      s[t][3] = fast_exp2(s[t][3] - ref1);
    }
    if (__any_sync(0xffffffffu, up0 || up1)) {
#pragma unroll
      for (int n = 0; n < MT_O; ++n) {
        o[n][0] *= al0; o[n][1] *= al1;
        o[n][2] *= al0; o[n][3] *= al1;
      }
      ol[0] *= al0; ol[1] *= al1; ol[2] *= al0; ol[3] *= al1;
    }
    // O^T += V^T P^T with the weights rounded to bf16 once; the all-ones A sums those weights
    const uint32_t ones[4] = {kOnesBf16x2, kOnesBf16x2, kOnesBf16x2, kOnesBf16x2};
#pragma unroll
    for (int kk = 0; kk < MT_S; ++kk) {
      const uint32_t b0 = movmatrix_trans(pack_bf16x2(s[kk][0], s[kk][1]));  // keys 2c, 2c+1
      const uint32_t b1 = movmatrix_trans(pack_bf16x2(s[kk][2], s[kk][3]));  // keys 2c+8, 2c+9
      mma_16816(ol, ones, b0, b1);
#pragma unroll
      for (int cb = 0; cb < MT_O; ++cb) {
        // matrices: keys 0-7 / 8-15 of this k-step (mat >> 1) x columns + 0-7 / + 8-15 (mat & 1)
        const int key = grp * KPW + kk * 16 + rr + ((mat >> 1) ? 8 : 0);
        uint32_t a[4];
        ldsm_x4_trans(swz_bytes(vbase, key, cb * 32 + (mat & 1) * 16), a[0], a[1], a[2], a[3]);
        mma_16816(o[cb], a, b0, b1);
      }
    }
  }

  // Publish this warp's state (the group's heads 0..7) to the combine scratch: output column
  // 16 b + r holds c0 / c1, column 16 b + r + 8 holds c2 / c3.
  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
    const int r = lane >> 2, h0 = (lane & 3) * 2;
    float* row0 = sh.comb_o + (warp * kCombRows + h0) * comb_row_floats(D);
    float* row1 = row0 + comb_row_floats(D);
#pragma unroll
    for (int b = 0; b < MT_O; ++b) {
      row0[b * 16 + r] = o[b][0];
      row0[b * 16 + r + 8] = o[b][2];
      row1[b * 16 + r] = o[b][1];
      row1[b * 16 + r + 8] = o[b][3];
    }
    if (r == 0) {
      sh.comb_ml[warp * kCombRows + h0] = make_float2(m[0], ol[0]);
      sh.comb_ml[warp * kCombRows + h0 + 1] = make_float2(m[1], ol[1]);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        ws[w] = w;
        rs[w] = hr;
      }
      return NW;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// CUDA-core consumer (G <= 7; over fp8 codes only when that path is forced). Warp w takes keys
// [KPW w, KPW (w + 1)) of every tile (KPW = 64 / NW, 16 or 8); lane owns DPL = D/32 consecutive
// columns of q, K, V and the output. EB: the cache's bytes per element (fp8 codes are widened
// exactly on load).
// ---------------------------------------------------------------------------------------------
template <int D, int G, int NW, int EB = 2>
struct CcConsumer {
  static constexpr int kWarps = NW;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = 1;
  static constexpr bool kSharedQ = false;
  static constexpr int kCombRows = 8;   // head rows per warp (G <= 7)
  static constexpr int DPL = D / 32;
  static constexpr int KPW = kTileKeys / NW;
  static_assert(KPW == 16 || KPW == 8, "the reduce-scatter below handles 8 or 16 keys per warp");
  // after the reduce-scatter, lane l holds the dot product of key l >> kLaneShift
  static constexpr int kLaneShift = KPW == 16 ? 1 : 2;
  static constexpr int kSame = 1 << kLaneShift;  // lanes holding the same key

  float qf[G][DPL];
  float o[G][DPL];
  float m[G], l[G];

  __device__ __forceinline__ void begin_segment(const DecodeParams& P, int bi, int j, int lane) {
    const __nv_bfloat16* qb = P.q + (static_cast<size_t>(bi) * P.h + static_cast<size_t>(j) * G) * D;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        qf[hh][e] = __bfloat162float(qb[hh * D + lane * DPL + e]);
        o[hh][e] = 0.f;
      }
      m[hh] = -INFINITY;
      l[hh] = 0.f;
    }
  }

  __device__ __forceinline__ void load_row(uint32_t base, int key, int lane, float (&f)[DPL]) const {
    const int c = lane * DPL * EB;  // byte column
    const uint32_t addr = swz_bytes(base, key, c & ~15) + (c & 15);
    if constexpr (EB == 1) {
      static_assert(DPL == 4, "fp8 rows of 128 columns: four codes per lane");
      uint32_t x, lo, hi;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(addr));
      e4m3x4_to_f16x2x2(x, lo, hi);
      const float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else if constexpr (DPL == 4) {
      uint32_t x, y;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(addr));
      const __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x);
      const __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&y);
      f[0] = __low2float(a); f[1] = __high2float(a);
      f[2] = __low2float(c); f[3] = __high2float(c);
    } else {
      uint32_t x;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(addr));
      const __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x);
      f[0] = __low2float(a); f[1] = __high2float(a);
    }
  }

  // Sum v[0..KPW-1] (one partial per key) over the 32 lanes; lane l ends with the full sum for
  // key l >> kLaneShift (the kSame lanes of a key hold the same value). Each exchange level halves
  // the values a lane keeps, so KPW keys cost KPW - 1 + kLaneShift shuffles instead of 5 KPW.
  __device__ __forceinline__ static float reduce_scatter(float (&v)[KPW], int lane) {
    float cur[KPW];
#pragma unroll
    for (int i = 0; i < KPW; ++i) cur[i] = v[i];
#pragma unroll
    for (int lvl = 0; (KPW >> lvl) > 1; ++lvl) {
      const int half = (KPW >> lvl) / 2;
      const int off = 16 >> lvl;
      const bool up = lane & off;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? cur[i] : cur[i + half];
        const float keep = up ? cur[i + half] : cur[i];
        cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    float r = cur[0];
#pragma unroll
    for (int off = kSame / 2; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
  }

  // `nvalid` = rows of this warp's 16 keys below the sequence length (warp-uniform, 0..16).
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int warp, int lane,
                                       int nvalid, float scale_log2) {
    const int key0 = warp * KPW;
    float kf[KPW][DPL];
#pragma unroll
    for (int kk = 0; kk < KPW; ++kk) {
      if (kk < nvalid) {
        load_row(kbase, key0 + kk, lane, kf[kk]);
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) kf[kk][e] = 0.f;
      }
    }
    const bool mine_valid = (lane >> kLaneShift) < nvalid;
    float p[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float part[KPW];
#pragma unroll
      for (int kk = 0; kk < KPW; ++kk) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc = fmaf(qf[hh][e], kf[kk][e], acc);
        part[kk] = acc;
      }
      const float dot = reduce_scatter(part, lane);
      const float s = mine_valid ? dot * scale_log2 : -INFINITY;
      float mx = s;
#pragma unroll
      for (int off = kSame; off <= 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[hh], mx);
      const float ref = (mn == -INFINITY) ? 0.f : mn;
      const float al = fast_exp2(m[hh] - ref);
      m[hh] = mn;
      p[hh] = fast_exp2(s - ref);
      l[hh] = l[hh] * al + ((lane & (kSame - 1)) ? 0.f : p[hh]);
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[hh][e] *= al;
    }
    // O += P V over the valid keys (p for key kk sits in lanes kk * kSame .. kk * kSame + kSame - 1)
#pragma unroll
    for (int kk = 0; kk < KPW; ++kk) {
      if (kk < nvalid) {
        float vf[DPL];
        load_row(vbase, key0 + kk, lane, vf);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float pk = __shfl_sync(0xffffffffu, p[hh], kk * kSame);
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[hh][e] = fmaf(pk, vf[e], o[hh][e]);
        }
      }
    }
  }

  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float lsum = l[hh];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      float* row = sh.comb_o + (warp * kCombRows + hh) * comb_row_floats(D);
#pragma unroll
      for (int e = 0; e < DPL; ++e) row[lane * DPL + e] = o[hh][e];
      if (lane == 0) sh.comb_ml[warp * kCombRows + hh] = make_float2(m[hh], lsum);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int w = 0; w < NW; ++w) { ws[w] = w; rs[w] = hr; }
      return NW;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// CUDA-core consumer for G <= 7 (automatically G <= 2), lanes owning keys (bf16 caches). Eight warps form two tile groups
// of four; a group takes every other tile of the CTA's range, so each group has two of the four
// stages (one being computed, one loading), and each warp 16 of a tile's 64 keys.
// In S = Q K^T each key belongs to two lanes, l and l + 16, which form the dot product over the
// lower and the upper half of the columns (the key's row from the stage in 16-byte loads, q from
// shared memory in fp32, every half-warp reading one address) and add the halves with one
// shuffle. The softmax takes one max over the warp's keys per head and tile; each lane keeps a
// partial sum over its key, reduced across the warp only when the segment's state is published.
// In O += P V each lane owns D/32 output columns and takes the keys' weights from a per-warp row
// in shared memory (written once per tile, read four keys at a time). The products run as packed
// fp32 pairs (fma.rn.f32x2): in S the two lanes of a pair sum the even and the odd columns, in
// P V the even and the odd keys; each pair is added up once, at the end of the tile (S) or of the
// segment (O).
// ---------------------------------------------------------------------------------------------
template <int D, int G>
struct CcConsumer2 {
  static constexpr int kWarps = 8;
  static constexpr int kRingBytes = mqa::kRingBytes;  // the stage ring
  static constexpr int kCtasPerSm = 1;
  static constexpr int kTileGroups = 2;
  static constexpr bool kSharedQ = true;
  static constexpr int kCombRows = 8;   // head rows per warp (G <= 7)
  static constexpr int DPL = D / 32;    // output columns per lane
  static constexpr int kKeys = kTileKeys * kTileGroups / kWarps;  // keys per warp and tile
  static constexpr int QH = D / 2;      // columns per half-warp in S
  static_assert(G <= kMaxCcHeads && (D == 64 || D == 128), "CUDA-core consumer shapes");
  static_assert(kKeys == kCcWarpKeys, "two lanes per key");
  static constexpr int kPvUnroll = G >= 6 ? 2 : 4;  // groups of four keys (more spills at G >= 6)

  uint64_t o2[G][DPL];  // O columns, as (even keys, odd keys) partial pairs
  float m[G];           // running reference, the same in every lane
  float l[G];           // this lane's share of the running sum (its key; lanes l, l + 16 agree)
  uint32_t qs;          // shared-window address of the staged q (explicit ld.shared: a generic
                        // pointer would make every q read wait like a global load)
  uint32_t pw;          // shared-window address of this warp's key weights [G][kKeys]

  // Stage q of segment (bi, j) in shared memory as fp32 (all consumer threads; the caller
  // synchronises the consumer warps before the first tile).
  __device__ __forceinline__ void begin_segment(const DecodeParams& P, const SharedLayout& sh,
                                                int bi, int j, int lane) {
    qs = smem_addr(sh.q_f32);
    pw = smem_addr(sh.p_cc) + (threadIdx.x >> 5) * kMaxCcHeads * kKeys * 4;
    const __nv_bfloat16* qb = P.q + row_offset(P, bi, j, 0, D);  // the group's G heads, adjacent
    for (int e = threadIdx.x; e < G * D; e += kWarps * 32)
      sh.q_f32[cc_q_index(D, e / D, e % D)] = __bfloat162float(qb[e]);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) o2[hh][e] = 0ull;
      m[hh] = -INFINITY;
      l[hh] = 0.f;
    }
  }

  // bf16 pair -> two floats (exact)
  __device__ __forceinline__ static float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ __forceinline__ static float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

  // One tile: this warp's keys are gw * 16 .. gw * 16 + 15 of the tile; `nvalid` of them (warp-
  // uniform, 0..16) lie below the sequence length.
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int gw, int lane,
                                       int nvalid, float scale_log2) {
    const int kl = lane & 15, dh = lane >> 4;
    const int key = gw * kKeys + kl;
    const uint32_t qh = qs + cc_q_index(D, 0, dh * QH) * 4;
    uint64_t acc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) acc[hh] = 0ull;
    // a few 8-column chunks at a time: unrolled further, the q reads of all heads stay live
#pragma unroll 2
    for (int c = 0; c < QH / 8; ++c) {
      uint32_t w0, w1, w2, w3;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                   : "r"(swz(kbase, key, dh * QH + c * 8)));
      const uint64_t k01 = pack_f32x2(lo_f(w0), hi_f(w0)), k23 = pack_f32x2(lo_f(w1), hi_f(w1));
      const uint64_t k45 = pack_f32x2(lo_f(w2), hi_f(w2)), k67 = pack_f32x2(lo_f(w3), hi_f(w3));
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        uint64_t q01, q23, q45, q67;
        const uint32_t qa = qh + (hh * cc_q_row_floats(D) + c * 8) * 4;
        asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(q01), "=l"(q23) : "r"(qa));
        asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(q45), "=l"(q67) : "r"(qa + 16));
        uint64_t a = acc[hh];
        a = fma_f32x2(q01, k01, a);
        a = fma_f32x2(q23, k23, a);
        a = fma_f32x2(q45, k45, a);
        a = fma_f32x2(q67, k67, a);
        acc[hh] = a;
      }
    }
    const bool mine_valid = kl < nvalid;
    float p[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float part = sum_f32x2(acc[hh]);
      part += __shfl_xor_sync(0xffffffffu, part, 16);  // both halves of the columns
      const float sc = mine_valid ? part * scale_log2 : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[hh], mx);
      const float ref = (mn == -INFINITY) ? 0.f : mn;
      const float al = fast_exp2(m[hh] - ref);
      m[hh] = mn;
      p[hh] = fast_exp2(sc - ref);  // 0 for keys at or beyond the length
      l[hh] = l[hh] * al + p[hh];
      const uint64_t al2 = pack_f32x2(al, al);
#pragma unroll
      for (int e = 0; e < DPL; ++e) o2[hh][e] = mul_f32x2(o2[hh][e], al2);
    }
    // the weights to this warp's rows (the previous tile's reads of them are done)
    __syncwarp();
    if (dh == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(pw + (hh * kKeys + kl) * 4), "f"(p[hh])
                     : "memory");
    }
    __syncwarp();
    // O += P V over the valid keys, four at a time
    if (nvalid == kKeys) {
#pragma unroll(kPvUnroll)
      for (int kq = 0; kq < kKeys; kq += 4) add_keys(vbase, gw, lane, kq, 4);
    } else {
      for (int kq = 0; kq < nvalid; kq += 4) add_keys(vbase, gw, lane, kq, nvalid - kq);
    }
  }

  // keys kq .. kq + 3 of the warp, the first `nv` (>= 1) of them valid; a row at or beyond the
  // length may hold anything, NaN included, so it is not read (its weight is 0)
  __device__ __forceinline__ void add_keys(uint32_t vbase, int gw, int lane, int kq, int nv) {
    const int d0 = lane * DPL;
    uint32_t x[4], y[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      x[r] = 0u;
      y[r] = 0u;
      const uint32_t a = swz(vbase, gw * kKeys + kq + r, d0 & ~7) + (d0 & 7) * 2;
      if (r < nv) {
        if constexpr (DPL == 4)
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x[r]), "=r"(y[r]) : "r"(a));
        else
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x[r]) : "r"(a));
      }
    }
    uint64_t va[DPL], vb[DPL];  // column e of keys (kq, kq + 1) and (kq + 2, kq + 3)
    va[0] = pack_f32x2(lo_f(x[0]), lo_f(x[1]));
    va[1] = pack_f32x2(hi_f(x[0]), hi_f(x[1]));
    vb[0] = pack_f32x2(lo_f(x[2]), lo_f(x[3]));
    vb[1] = pack_f32x2(hi_f(x[2]), hi_f(x[3]));
    if constexpr (DPL == 4) {
      va[2] = pack_f32x2(lo_f(y[0]), lo_f(y[1]));
      va[3] = pack_f32x2(hi_f(y[0]), hi_f(y[1]));
      vb[2] = pack_f32x2(lo_f(y[2]), lo_f(y[3]));
      vb[3] = pack_f32x2(hi_f(y[2]), hi_f(y[3]));
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      uint64_t p01, p23;
      asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];"
                   : "=l"(p01), "=l"(p23)
                   : "r"(pw + (hh * kKeys + kq) * 4));
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        o2[hh][e] = fma_f32x2(p01, va[e], o2[hh][e]);
        o2[hh][e] = fma_f32x2(p23, vb[e], o2[hh][e]);
      }
    }
  }

  __device__ __forceinline__ void publish(const SharedLayout& sh, int warp, int lane) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float lsum = l[hh];  // over the 16 keys (lanes l and l + 16 hold the same key's share)
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      float* row = sh.comb_o + (warp * kCombRows + hh) * comb_row_floats(D);
#pragma unroll
      for (int e = 0; e < DPL; ++e) row[lane * DPL + e] = sum_f32x2(o2[hh][e]);
      if (lane == 0) sh.comb_ml[warp * kCombRows + hh] = make_float2(m[hh], lsum);
    }
  }

  struct Rows {
    __device__ __forceinline__ int operator()(int hr, int* ws, int* rs) const {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) { ws[w] = w; rs[w] = hr; }
      return kWarps;
    }
  };
};

// ---------------------------------------------------------------------------------------------
// The kernel. `Consumer` is MmaConsumerT<D, NW>, MmaConsumer<D, WM, NW>, MmaConsumerF8T<D, NW, TG>,
// MmaConsumerF8<D, WM, NW, TG>, CcConsumer2<D, G> or CcConsumer<D, G, NW, EB>; EB: the cache's
// bytes per element (2 bf16, 1 fp8). The consumer also sets the stage ring's size and the CTAs
// per SM the kernel is built for.
// ---------------------------------------------------------------------------------------------
template <int D, int EB, class Consumer, bool kTensorCores, int WM>
__global__ void __launch_bounds__(threads_of(Consumer::kWarps), Consumer::kCtasPerSm)
    decode_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const DecodeParams P) {
  constexpr int RB = Consumer::kRingBytes;
  using Geo = Geometry<D, EB, RB>;
  constexpr int kStages = Geo::kStages;
  constexpr int NW = Consumer::kWarps;
  constexpr int CR = Consumer::kCombRows;
  constexpr int kThreads = threads_of(NW);
  extern __shared__ uint8_t smem_raw[];
  SharedLayout sh = carve_shared<D, EB, NW, CR, RB>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Programmatic dependent launch (when the host asked for it): this kernel reads its inputs at
  // once. Without early writes it writes global memory (outputs, partial states, counters,
  // appended cache rows) only after pdl_wait(), once the kernel ahead has finished. In both
  // modes the launch-order warp below lets the next launch be scheduled after its own wait.

  // ---- barriers, then the tiles of every sequence and their prefix ---------------------------
  __shared__ uint32_t chunk_tiles[kThreads + 1];
  if (tid == 0) {
    *sh.abort = 0;
    *sh.merge = 0;
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&sh.full[st], 1);
      mbar_init(&sh.empty[st], NW / Consumer::kTileGroups);  // the warps of one tile group
    }
    mbar_init(sh.cbar, NW * 32);
    mbar_init(sh.stall, 1);
    fence_barrier_init();
  }
  build_tile_prefix<kThreads>(P, sh, chunk_tiles);

  zero_invalid_sequences<D>(P, kThreads);
  if (P.pos != nullptr) append_uncovered_rows<D, EB>(P, kThreads);

  const unsigned long long W = sh.tix.total();
  const unsigned long long x0 = W * blockIdx.x / P.num_ctas;
  const unsigned long long x1 = W * (blockIdx.x + 1) / P.num_ctas;
  if (x0 >= x1) {
    // a CTA with no tiles still waits for the kernel ahead before it exits, so that this grid
    // never completes (nor lets the next launch start) before that kernel has
    pdl_wait();
    return;
  }
  const int ntiles = static_cast<int>(x1 - x0);
  const uint32_t stages_base = smem_addr(sh.stages);
  constexpr uint32_t kStageBytes = Geo::kStageBytes;
  constexpr uint32_t kKvBytes = Geo::kKvBytes;

  if constexpr (NW == 8) {
    if (warp >= NW) setmaxnreg_dec<kProducerRegs>();
    else setmaxnreg_inc<kConsumerRegs>();
  }
  if (warp >= NW) {
    // ================================ producer ================================================
    // warps NW and NW + 2 issue alternate tiles (a tile takes two or four copies from contiguous
    // caches, up to 2 * 64 / page_size from paged ones), so one warp's issue rate does not bound
    // the CTA
    const bool paged = P.page_table != nullptr;
    const int np = paged ? kPagedProducers : kContiguousProducers;
    if (warp == NW || (np == 2 && warp == NW + 2)) {
      const int pi = warp == NW ? 0 : 1;
      if (paged)
        produce_tiles_paged_any<D, EB, RB>(&tm_k, &tm_v, P, sh, x0, ntiles, lane, np, pi);
      else
        produce_tiles<D, EB, RB>(&tm_k, &tm_v, P, sh, x0, ntiles, lane, np, pi);
    } else if (warp == NW + 1 && lane == 0) {
      // ============================ launch order ==============================================
      pdl_wait();
      pdl_launch_dependents();
    }
    return;
  }

  // ================================== consumers ================================================
  Consumer cons;
  // tile groups: warp group tg owns the tiles k with k % TG == tg (TG = 1: every warp, every tile)
  constexpr int TG = Consumer::kTileGroups;
  constexpr int WPG = NW / TG;  // warps per tile group
  static_assert(TG == 1 || kTensorCores || Consumer::kSharedQ, "tile groups of this consumer");
  // Each stage must always serve the same tile group, which takes its uses in order: a group
  // that could wait on a stage two uses ahead would see the parity of the use before it.
  static_assert(kStages % TG == 0, "stages per tile group");
  // and each stage to one paged producer warp (its drain relies on it)
  static_assert(kStages % kPagedProducers == 0 && kStages % kContiguousProducers == 0,
                "stages per producer");
  const int tg = warp / WPG;
  const int gw = warp % WPG;
  const int grp = kTensorCores ? gw / WM : warp;
  const int mi = kTensorCores ? gw % WM : 0;
  constexpr int kGroupKeys = kTensorCores ? kTileKeys * WM / WPG : kTileKeys / WPG;
  uint32_t cphase = 0;
  TileCursor cur;
  cur.start(x0, sh.tix);
  int L = 0;
  bool began_at_zero = false;
  bool after_dep = false;  // pdl_wait() done: global writes allowed
  if (P.debug_stall == 1 && !mbar_wait_bounded(sh.stall, 0, P.timeout_ns, sh.abort)) {
    if (!*sh.abort) give_up(sh, kSiteStall, 0);
    return;
  }
  for (int k = 0; k < ntiles; ++k) {
    const int st = k % kStages;
    const bool mine = TG == 1 || k % TG == tg;
    // a segment's q and length are read before its first tile is waited for, so that their
    // global-memory latency overlaps the tile's copy (every warp is past the previous segment's
    // end: that end synchronised the consumer warps)
    if (k == 0 || cur.tile == 0) {
      L = __ldg(P.seq_lens + cur.bi);
      began_at_zero = (cur.tile == 0);
      if constexpr (kTensorCores) {
        cons.begin_segment(P, cur.bi, cur.j, mi, lane);
      } else if constexpr (Consumer::kSharedQ) {
        // every consumer warp is at this segment start (the last segment's end synchronised
        // them); q is staged in shared memory before any warp's first tile of the segment
        cons.begin_segment(P, sh, cur.bi, cur.j, lane);
        if (!consumer_sync(sh, cphase, P.timeout_ns)) {
          if (!*sh.abort) give_up(sh, kSiteConsumerSync, k);
          return;
        }
      } else {
        cons.begin_segment(P, cur.bi, cur.j, lane);
      }
    }
    if (mine && !mbar_wait_bounded(&sh.full[st], (k / kStages) & 1, P.timeout_ns, sh.abort)) {
      if (!*sh.abort) give_up(sh, kSiteConsumerFull, k);
      return;
    }
    const int tile_start = cur.tile * kTileKeys;
    const int valid = min(L - tile_start, kTileKeys);  // >= 1
    const uint32_t kbase = stages_base + st * kStageBytes;
    const uint32_t vbase = kbase + kKvBytes;
    if (!mine) {
      // another tile group's tile: only the segment bookkeeping below
    } else if constexpr (kTensorCores) {
      // V rows at or beyond the length may hold anything (NaN included) and 0 * NaN = NaN on
      // the tensor cores: zero this group's invalid V rows before P V reads them.
      const int g0 = grp * kGroupKeys;
      if (valid < g0 + kGroupKeys) {
        uint8_t* vst = sh.stages + st * kStageBytes + kKvBytes;
        const int first = max(valid, g0);
        const int rows = g0 + kGroupKeys - first;
        constexpr int chunks_per_row = Geo::kRowBytes / 16;
        for (int c = lane; c < rows * chunks_per_row; c += 32) {
          const int key = first + c / chunks_per_row;
          const int ch = c % chunks_per_row;
          const int half = ch >> 3, sub = ch & 7;
          *reinterpret_cast<uint4*>(vst + half * kTileKeys * kSwizzleRowBytes +
                                    key * kSwizzleRowBytes + sub * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // the consumer masks by the rows left from this tile's start (not capped at the tile), so
      // that a row's causal lag applies at the sequence's end only
      cons.tile(kbase, vbase, grp, lane, L - tile_start, P.scale_log2);
    } else {
      const int nvalid = max(0, min(valid - gw * kGroupKeys, kGroupKeys));
      cons.tile(kbase, vbase, gw, lane, nvalid, P.scale_log2);
    }
    if (mine) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[st]);
    }

    const bool seg_end = (cur.tile == cur.nt - 1);
    if (seg_end || k == ntiles - 1) {
      const bool complete = began_at_zero && seg_end;
      const int seg = cur.bi * P.g + cur.j;
      cons.publish(sh, warp, lane);
      if (!consumer_sync(sh, cphase, P.timeout_ns)) {
        if (!*sh.abort) give_up(sh, kSiteConsumerSync, k);
        return;
      }
      if (!after_dep) {
        if (!P.early_writes) pdl_wait();
        after_dep = true;
      }
      combine_and_store<D, NW, CR>(P, sh, cur.bi, cur.j, complete,
                                   static_cast<int>(blockIdx.x) + seg, typename Consumer::Rows{});
      if (!complete) __threadfence();  // this CTA's partial is visible before it is counted
      if (!consumer_sync(sh, cphase, P.timeout_ns)) {
        if (!*sh.abort) give_up(sh, kSiteConsumerSync, k);
        return;
      }
      if (!complete && !finish_split_segment<D, NW, CR>(P, sh, cphase, cur, W)) {
        if (!*sh.abort) give_up(sh, kSiteConsumerSync, k);
        return;
      }
    }
    cur.advance(sh.tix);
  }
}

}  // namespace mqa
