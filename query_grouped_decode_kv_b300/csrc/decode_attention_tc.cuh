// decode_attention_tc.cuh -- grouped decode attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory) for sm_103a.
//
// Same definition, work split, fused append and split merge as decode_attention.cuh
// ("分组查询注意力（GQA）与多查询注意力（MQA）深度实战", ybb.press, §五: O_i = softmax_t(scale q_i.K_{j,t})
// V_{j,t} with j = i / G); only the inner products and the softmax are organised differently.
// The G query heads of a KV head are the rows of a 128-row MMA tile (rows >= G hold zeros):
//
//   S = Q K^T          M = 128 head rows, N = 64 keys, K = d_h; A = Q and B = the K tile, both
//                      from shared memory (128-byte swizzle); S in tensor memory, fp32
//   softmax            one thread per head row: it loads its 64 scores from tensor memory, so row
//                      maxima and sums need no shuffles; P (bf16) goes back into tensor memory
//                      over the first half of S's columns
//   O += P V           M = 128, N = d_h, K = 64 keys; A = P from tensor memory, B = the V tile
//                      from shared memory (N-major); O in tensor memory, fp32
//
// Warp roles (192 threads): warps 0-3 run the softmax and the epilogue (thread t owns head row
// t, tensor-memory lane t); warp 4 is the bulk-copy producer shared with the other kernel; one
// lane of warp 5 issues the MMAs, and warp 5 owns the tensor-memory allocation. S is double
// buffered: the MMA of tile k+1's scores runs while the softmax of tile k does.
//
// Online softmax with a lazy reference: a row's probabilities are exp2(s - m_ref), where m_ref is
// the row's maximum when the segment started or when it was last raised; it is raised, and O and
// the running sum rescaled, only when a new maximum exceeds m_ref by more than kRescaleLog2, so
// the probabilities stay below 2^kRescaleLog2 and O is rarely touched. (The merge of split
// segments takes any reference, so partial states keep theirs.)
//
// Every wait is bounded in time; on expiry the kernel latches MQA_ERR_TIMEOUT, and warp 5 waits
// (bounded) for its MMAs and for the softmax warps before it frees the tensor memory.
#pragma once

#include "decode_attention.cuh"

namespace mqa {

constexpr int kTcThreads = 192;
constexpr int kTcRows = 128;          // MMA M: head rows
constexpr int kTcTmemCols = 256;      // S: 2 x 64 columns; O: d_h <= 128 columns
constexpr int kTcMergeRows = 4;       // rows per warp of merge scratch (see merge_split_segment)
constexpr float kRescaleLog2 = 8.f;

__host__ __device__ constexpr int tc_q_bytes(int D) { return kTcRows * D * 2; }
__host__ __device__ constexpr int tc_barrier_count() { return 2 * kStages + 1 + 9; }
__host__ __device__ constexpr int tc_smem_fixed_bytes(int D) {
  return kStages * stage_bytes(D) + tc_q_bytes(D) + 4 * kTcMergeRows * comb_row_floats(D) * 4 +
         4 * kTcMergeRows * 8 + tc_barrier_count() * 8 + 32;
}
__host__ __device__ constexpr size_t tc_smem_bytes(int D, int b) {
  return 1024 + static_cast<size_t>(tc_smem_fixed_bytes(D)) + static_cast<size_t>(b + 1) * 4;
}

struct TcShared {
  SharedLayout base;   // stage ring, merge scratch, full/empty/cbar barriers, flags, tile prefix
  uint8_t* q;          // [D/64][128 rows][128 B], 128-byte swizzle, 1024-aligned
  uint64_t* s_full;    // [2] S of the tile in buffer k % 2 is complete (MMA commit)
  uint64_t* p_full;    // [2] P of the tile in buffer k % 2 is in tensor memory (128 threads)
  uint64_t* pv_done;   // [2] O += P V of the tile with parity k % 2 is complete (MMA commit)
  uint64_t* q_full;    // Q of the next segment is in shared memory (128 softmax threads)
  uint64_t* tmem_done; // the softmax warps no longer touch tensor memory (128 arrivals)
  uint64_t* drain;     // every MMA issued so far is complete (MMA commit, at exit)
  uint32_t* tmem_base; // written by tcgen05.alloc
};

template <int D>
__device__ __forceinline__ TcShared carve_tc_shared(uint8_t* raw) {
  TcShared t;
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  t.base.stages = p;
  p += kStages * stage_bytes(D);
  t.q = p;
  p += tc_q_bytes(D);
  t.base.comb_o = reinterpret_cast<float*>(p);
  p += 4 * kTcMergeRows * comb_row_floats(D) * 4;
  t.base.comb_ml = reinterpret_cast<float2*>(p);
  p += 4 * kTcMergeRows * 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  t.base.full = bars;
  t.base.empty = bars + kStages;
  t.base.cbar = bars + 2 * kStages;
  t.s_full = bars + 2 * kStages + 1;
  t.p_full = t.s_full + 2;
  t.pv_done = t.p_full + 2;
  t.q_full = t.pv_done + 2;
  t.tmem_done = t.q_full + 1;
  t.drain = t.tmem_done + 1;
  p += tc_barrier_count() * 8;
  t.base.abort = reinterpret_cast<volatile int*>(p);
  t.base.merge = t.base.abort + 1;
  t.tmem_base = reinterpret_cast<uint32_t*>(p + 8);
  p += 32;
  t.base.pre = reinterpret_cast<uint32_t*>(p);
  return t;
}

// Q of segment (bi, j) into head rows 0 .. G-1 of the swizzled Q tile (128 consumer threads).
template <int D>
__device__ __forceinline__ void tc_write_q(const DecodeParams& P, const TcShared& sh, int bi,
                                           int j) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const uint4* src = reinterpret_cast<const uint4*>(
      P.q + (static_cast<size_t>(bi) * P.h + static_cast<size_t>(j) * P.G) * D);
  for (int e = threadIdx.x; e < P.G * CH; e += 128) {
    const int r = e / CH, c = e - (e / CH) * CH;
    const int half = c >> 3, sub = c & 7;
    *reinterpret_cast<uint4*>(sh.q + half * (kTcRows * kSwizzleRowBytes) + r * kSwizzleRowBytes +
                              ((sub ^ (r & 7)) << 4)) = __ldg(src + e);
  }
}

// ---------------------------------------------------------------------------------------------
// MMA issue (one lane of warp 5). Tile k uses stage k % kStages and S buffer k % 2.
// ---------------------------------------------------------------------------------------------
template <int D>
struct TcMma {
  static constexpr uint32_t kIdescS = umma_idesc_bf16_f32(kTcRows, kTileKeys, false);
  static constexpr uint32_t kIdescO = umma_idesc_bf16_f32(kTcRows, D, true);
  uint32_t stages, q, tmem;

  // S(k) = Q K_k^T: K-steps of 16 along d_h; both operands K-major, 8-row groups 1024 B apart,
  // the second 64-column half of a row 16 KB (Q) or 8 KB (K) further on.
  __device__ __forceinline__ void scores(int k) const {
    const uint32_t kst = stages + (k % kStages) * stage_bytes(D);
    const uint32_t d_tmem = tmem + (k & 1) * kTileKeys;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk & 3) * 32;
      const uint64_t a = sw128_desc(q + (kk >> 2) * (kTcRows * kSwizzleRowBytes) + off, 0, 1024);
      const uint64_t b = sw128_desc(kst + (kk >> 2) * (kTileKeys * kSwizzleRowBytes) + off, 0,
                                    1024);
      umma_ss(d_tmem, a, b, kIdescS, kk > 0 ? 1u : 0u);
    }
  }
  // O (+)= P(k) V_k: K-steps of 16 keys; P from tensor memory (16 keys = 8 columns of bf16
  // pairs), V N-major: 64-column halves 8 KB apart (leading offset), 8-key groups 1024 B apart.
  __device__ __forceinline__ void values(int k, bool overwrite) const {
    const uint32_t vst = stages + (k % kStages) * stage_bytes(D) + stage_bytes(D) / 2;
    const uint32_t p_tmem = tmem + (k & 1) * kTileKeys;
    const uint32_t o_tmem = tmem + 2 * kTileKeys;
#pragma unroll
    for (int kk = 0; kk < kTileKeys / 16; ++kk) {
      const uint64_t b = sw128_desc(vst + kk * 16 * kSwizzleRowBytes,
                                    kTileKeys * kSwizzleRowBytes, 1024);
      umma_ts(o_tmem, p_tmem + kk * 8, b, kIdescO, (overwrite && kk == 0) ? 0u : 1u);
    }
  }
};

// The P and PV barriers alternate between two instances, tile k on instance k % 2, so that no
// waiter can be two phases away from the one it asks for (a parity wait cannot tell those apart):
//  - the issuer waits for P(k) after it has issued S(k+1), so the softmax warps may already have
//    finished P(k+1); P(k+2) needs S(k+2), which is issued only after P(k) was seen;
//  - within a segment S(k) is issued before O += P(k-1) V, so when the softmax warps hold S(k) the
//    PV of tile k-1 may still run while that of k-2 has finished (S(k)'s commit covers it); PV
//    of tile k+1 needs P(k+1), which they have not produced yet.
template <int D>
__device__ __forceinline__ void tc_issue_loop(const DecodeParams& P, const TcShared& sh,
                                              uint32_t tmem, unsigned long long x0, int ntiles) {
  const SharedLayout& b = sh.base;
  TcMma<D> mma{smem_addr(b.stages), smem_addr(sh.q), tmem};
  // S(kn) into buffer kn % 2 once its stage has landed and the P V product that last read that
  // buffer (tile kn - 2, its P aliases the buffer's first columns) has finished
  auto issue_scores = [&](int kn) -> bool {
    if (kn >= 2 && !mbar_wait_bounded(&sh.pv_done[kn & 1], ((kn - 2) >> 1) & 1, P.timeout_ns,
                                      b.abort)) {
      if (!*b.abort) give_up(b, kSiteMmaPv, kn);
      return false;
    }
    if (!mbar_wait_bounded(&b.full[kn % kStages], (kn / kStages) & 1, P.timeout_ns, b.abort)) {
      if (!*b.abort) give_up(b, kSiteMmaFull, kn);
      return false;
    }
    tc_fence_after_sync();
    mma.scores(kn);
    umma_commit(&sh.s_full[kn & 1]);
    return true;
  };
  TileCursor cur;
  cur.start(x0, b.pre, P.b, P.g);
  uint32_t qphase = 0;
  if (!mbar_wait_bounded(sh.q_full, 0, P.timeout_ns, b.abort)) {
    if (!*b.abort) give_up(b, kSiteMmaQ, 0);
    return;
  }
  if (!issue_scores(0)) return;
  for (int k = 0; k < ntiles; ++k) {
    TileCursor nxt = cur;
    nxt.advance(b.pre, P.b, P.g);
    const bool has_next = k + 1 < ntiles;
    const bool next_new = has_next && nxt.tile == 0;  // the next tile starts a segment
    // same segment: the next tile's scores run while the softmax of this one does
    if (has_next && !next_new && !issue_scores(k + 1)) return;
    if (!mbar_wait_bounded(&sh.p_full[k & 1], (k >> 1) & 1, P.timeout_ns, b.abort)) {
      if (!*b.abort) give_up(b, kSiteMmaP, k);
      return;
    }
    tc_fence_after_sync();
    mma.values(k, k == 0 || cur.tile == 0);
    umma_commit(&sh.pv_done[k & 1]);
    umma_commit(&b.empty[k % kStages]);
    if (next_new) {  // a new segment: its Q must be in place first
      ++qphase;
      if (!mbar_wait_bounded(sh.q_full, qphase & 1, P.timeout_ns, b.abort)) {
        if (!*b.abort) give_up(b, kSiteMmaQ, k + 1);
        return;
      }
      if (!issue_scores(k + 1)) return;
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------------------------
// Softmax and epilogue (warps 0-3; thread t = head row t = tensor-memory lane t).
// Returns false if a wait timed out.
// ---------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ bool tc_softmax_loop(const DecodeParams& P, const TcShared& sh,
                                                uint32_t tmem, unsigned long long x0, int ntiles,
                                                unsigned long long W) {
  const SharedLayout& b = sh.base;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = P.G;
  const bool warp_rows = warp * 32 < G;   // warp-uniform: this warp holds real head rows
  const bool my_row = tid < G;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_s = tmem + lane_base;                 // S / P buffers (+64 for the second)
  const uint32_t t_o = tmem + lane_base + 2 * kTileKeys; // O
  constexpr uint32_t kStageBytes = stage_bytes(D);
  uint32_t cphase = 0;

  // Q: the first segment's rows (rows >= G were zeroed in the prologue; each chunk of the tile has
  // exactly one writer, so no write here can land on another thread's)
  TileCursor cur;
  cur.start(x0, b.pre, P.b, P.g);
  tc_write_q<D>(P, sh, cur.bi, cur.j);
  fence_proxy_async_smem();
  mbar_arrive(sh.q_full);

  float m_ref = -INFINITY, l = 0.f;
  int L = 0;
  bool began_at_zero = false;
  for (int k = 0; k < ntiles; ++k) {
    const bool first = (k == 0 || cur.tile == 0);
    if (first) {
      L = __ldg(P.seq_lens + cur.bi);
      began_at_zero = (cur.tile == 0);
      m_ref = -INFINITY;
      l = 0.f;
    }
    const int valid = min(L - cur.tile * kTileKeys, kTileKeys);  // >= 1
    bool ok = mbar_wait_bounded(&sh.s_full[k & 1], (k >> 1) & 1, P.timeout_ns, b.abort);
    if (!ok && !*b.abort) give_up(b, kSiteSoftmaxS, k);
    if (!__all_sync(0xffffffffu, ok)) return false;
    tc_fence_after_sync();
    if (warp_rows) {
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(t_s + (k & 1) * kTileKeys, r0);
      tmem_ld_32x32b_x32(t_s + (k & 1) * kTileKeys + 32, r1);
      tmem_wait_ld();
      float s[kTileKeys];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = c < valid ? __uint_as_float(r0[c]) * P.scale_log2 : -INFINITY;
        s[c + 32] = c + 32 < valid ? __uint_as_float(r1[c]) * P.scale_log2 : -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kTileKeys; ++c) mx = fmaxf(mx, s[c]);
      float alpha = 1.f;
      bool raise = false;
      if (first) {
        m_ref = mx;
      } else if (mx > m_ref + kRescaleLog2) {
        raise = true;
        alpha = fast_exp2(m_ref - mx);
        m_ref = mx;
        l *= alpha;
      }
      if (__any_sync(0xffffffffu, raise)) {
        // O must hold P V of the previous tile before it is rescaled
        ok = mbar_wait_bounded(&sh.pv_done[(k - 1) & 1], ((k - 1) >> 1) & 1, P.timeout_ns,
                               b.abort);
        if (!ok && !*b.abort) give_up(b, kSiteSoftmaxPv, k);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(t_o + c, o);
        }
        tmem_wait_st();
      }
      // probabilities rounded to bf16 once: the same values feed P V and the running sum
      uint32_t pk[32];
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = round_bf16(fast_exp2(s[2 * i] - m_ref));
        const float p1 = round_bf16(fast_exp2(s[2 * i + 1] - m_ref));
        ps += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l += ps;
      tmem_st_32x32b_x32(t_s + (k & 1) * kTileKeys, pk);
      tmem_wait_st();
    }
    if (valid < kTileKeys) {
      // V rows at or beyond the length may hold anything (NaN included), and 0 * NaN = NaN in
      // the MMA: zero them. The stage's full barrier is complete (the scores read its K half);
      // waiting on it orders the bulk copy's writes before these.
      const int st = k % kStages;
      ok = mbar_wait_bounded(&b.full[st], (k / kStages) & 1, P.timeout_ns, b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteSoftmaxFull, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      uint8_t* vst = b.stages + st * kStageBytes + kStageBytes / 2;
      constexpr int CH = D / 8;
      for (int e = tid; e < (kTileKeys - valid) * CH; e += 128) {
        const int key = valid + e / CH, c = e - (e / CH) * CH;
        *reinterpret_cast<uint4*>(vst + (c >> 3) * (kTileKeys * kSwizzleRowBytes) +
                                  key * kSwizzleRowBytes + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    mbar_arrive(&sh.p_full[k & 1]);

    TileCursor nxt = cur;
    nxt.advance(b.pre, P.b, P.g);
    const bool has_next = k + 1 < ntiles;
    if (has_next && nxt.tile == 0) {
      // the next tile starts a segment; S(k) has finished reading this segment's Q
      tc_write_q<D>(P, sh, nxt.bi, nxt.j);
      fence_proxy_async_smem();
      mbar_arrive(sh.q_full);
    }

    const bool seg_end = (cur.tile == cur.nt - 1);
    if (seg_end || !has_next) {
      ok = mbar_wait_bounded(&sh.pv_done[k & 1], (k >> 1) & 1, P.timeout_ns, b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteEpiloguePv, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after_sync();
      const bool complete = began_at_zero && seg_end;
      const int seg = cur.bi * P.g + cur.j;
      const size_t slot = static_cast<size_t>(blockIdx.x) + seg;
      if (warp_rows) {
        const float inv_l = 1.f / l;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c, o);
          tmem_wait_ld();
          if (my_row && complete) {
            uint4* dst = reinterpret_cast<uint4*>(
                P.out + (static_cast<size_t>(cur.bi) * P.h + static_cast<size_t>(cur.j) * G +
                         tid) * D + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv_l,
                                __uint_as_float(o[8 * i + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv_l,
                                __uint_as_float(o[8 * i + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv_l,
                                __uint_as_float(o[8 * i + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv_l,
                                __uint_as_float(o[8 * i + 7]) * inv_l);
              dst[i] = v;
            }
          } else if (my_row) {
            uint4* dst = reinterpret_cast<uint4*>(P.part_o + (slot * G + tid) * D + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
        if (my_row && !complete) P.part_ml[slot * G + tid] = make_float2(m_ref, l);
      }
      if (!complete) __threadfence();  // this CTA's partial is visible before it is counted
      if (!consumer_sync(b, cphase, P.timeout_ns) ||
          (!complete &&
           !finish_split_segment<D, 4, kTcMergeRows>(P, b, cphase, cur.bi, cur.j, cur.nt, W))) {
        if (!*b.abort) give_up(b, kSiteConsumerSync, k);
        return false;
      }
    }
    cur = nxt;
  }
  return true;
}

// ---------------------------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v, const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  const TcShared sh = carve_tc_shared<D>(smem_raw);
  const SharedLayout& b = sh.base;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (warp == 5) {
    tmem_alloc(sh.tmem_base, kTcTmemCols);
    tmem_relinquish_alloc_permit();
  }
  __shared__ uint32_t part_sums[kTcThreads];
  if (tid == 0) {
    *b.abort = 0;
    *b.merge = 0;
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&b.full[st], 1);
      mbar_init(&b.empty[st], 1);   // one MMA commit frees a stage
    }
    mbar_init(b.cbar, 128);
    mbar_init(&sh.s_full[0], 1);
    mbar_init(&sh.s_full[1], 1);
    mbar_init(&sh.p_full[0], 128);
    mbar_init(&sh.p_full[1], 128);
    mbar_init(&sh.pv_done[0], 1);
    mbar_init(&sh.pv_done[1], 1);
    mbar_init(sh.q_full, 128);
    mbar_init(sh.tmem_done, 128);
    mbar_init(sh.drain, 1);
    fence_barrier_init();
  }
  // head rows G .. 127 of the Q tile stay zero for the whole launch (their S rows are ignored);
  // the CTA-wide barrier below orders these writes before any Q row is written or read
  {
    constexpr int CH = D / 8;
    const int first = P.G * CH, rows_total = kTcRows * CH;
    for (int e = first + tid; e < rows_total; e += kTcThreads) {
      const int r = e / CH, c = e - (e / CH) * CH;
      *reinterpret_cast<uint4*>(sh.q + (c >> 3) * (kTcRows * kSwizzleRowBytes) +
                                r * kSwizzleRowBytes + (((c & 7) ^ (r & 7)) << 4)) =
          make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before_sync();
  build_tile_prefix<kTcThreads>(P, b, part_sums);  // ends with a CTA-wide barrier
  tc_fence_after_sync();
  const uint32_t tmem = *sh.tmem_base;

  zero_invalid_sequences<D>(P, kTcThreads);
  if (P.pos != nullptr) append_uncovered_rows<D>(P, kTcThreads);

  const unsigned long long W = static_cast<unsigned long long>(P.g) * b.pre[P.b];
  const unsigned long long x0 = W * blockIdx.x / P.num_ctas;
  const unsigned long long x1 = W * (blockIdx.x + 1) / P.num_ctas;
  if (x0 >= x1) {
    if (warp == 5) tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  const int ntiles = static_cast<int>(x1 - x0);

  if (warp == 4) {
    produce_tiles<D>(&tm_k, &tm_v, P, b, x0, ntiles, lane);
    return;
  }
  if (warp == 5) {
    const volatile int never = 0;
    if (lane == 0) {
      tc_issue_loop<D>(P, sh, tmem, x0, ntiles);
      // every MMA issued has finished, and the softmax warps are done, before the columns go
      umma_commit(sh.drain);
      if (!mbar_wait_bounded(sh.drain, 0, P.timeout_ns, &never)) give_up(b, kSiteDrain, ntiles);
      if (!mbar_wait_bounded(sh.tmem_done, 0, 3 * P.timeout_ns, &never))
        give_up(b, kSiteTmemDone, ntiles);
    }
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  // warps 0-3
  tc_softmax_loop<D>(P, sh, tmem, x0, ntiles, W);  // a timed-out wait has recorded itself
  tc_fence_before_sync();
  mbar_arrive(sh.tmem_done);
}

}  // namespace mqa
