// decode_attention_tc.cuh -- grouped decode attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory) for sm_103a.
//
// Same definition, work split, fused append and split merge as decode_attention.cuh
// ("分组查询注意力（GQA）与多查询注意力（MQA）深度实战", ybb.press, §五: O_i = softmax_t(scale q_i.K_{j,t})
// V_{j,t} with j = i / G); only the inner products and the softmax are organised differently.
//
// Head rows and copies. The MMA tile has 128 rows; the G heads of the KV group, padded to
// GP in {16, 32, 64}, fill GP of them, and the tile holds C = 128 / GP copies of the group:
// row r = c * GP + h is head h (zero when h >= G) of copy c. All copies see the same scores, but
// copy c owns only the keys [c * OWN, (c + 1) * OWN) of each 64-key tile (OWN = 64 / C) and runs
// its own online softmax over them; the copies' states are merged (log-sum-exp) once per segment.
// Each thread owns one row, so the softmax of a tile costs OWN exponentials per thread, spread
// over all four SM sub-partitions, instead of 64 on the one sub-partition that holds the heads.
//
//   S = Q K^T          M = 128 rows, N = 64 keys, K = d_h; A = Q, B = the K tile, both from shared
//                      memory (128-byte swizzle); S in tensor memory, fp32
//   softmax            thread r loads its OWN scores, writes its bf16 probabilities into its row of
//                      a P buffer in tensor memory (the row's other columns stay zero)
//   O += P V           M = 128, N = d_h, K = 64 keys; A = P from tensor memory, B = the V tile
//                      from shared memory (N-major); O in tensor memory, fp32
//
// Tensor memory (512 columns): kTcBufs S buffers of 64 columns, kTcBufs P buffers of 32 columns
// (64 keys as bf16 pairs), and O. With four buffers the issuing thread runs the score MMAs up to
// three tiles ahead of the softmax.
//
// Shared memory holds separate rings of K and V tiles, as deep as shared memory allows (5 + 6
// tiles at d_h = 128). A K tile is done once its scores are, a V tile only once O += P V is,
// after the softmax; separate rings let the K copies run ahead, and the depth keeps enough
// copies in flight to cover the memory latency under full load (about 3 us).
//
// Warp roles (192 threads): warps 0-3 run the softmax and the epilogue (thread t = row t =
// tensor-memory lane t); warp 4 is the bulk-copy producer shared with the other kernel; one lane
// of warp 5 issues the MMAs, and warp 5 owns the tensor-memory allocation.
//
// Online softmax with a lazy reference: a row's probabilities are exp2(s - m_ref), where m_ref is
// the row's maximum when its segment started or when it was last raised; it is raised, and the
// row of O and the running sum rescaled, only when a new maximum exceeds m_ref by more than
// kLazyLog2. (Merges take any reference.)
//
// Every wait is bounded in time; on expiry the kernel records the wait, latches MQA_ERR_TIMEOUT,
// and warp 5 waits (bounded) for its MMAs and for the softmax warps before it frees the tensor
// memory.
#pragma once

#include "decode_attention.cuh"

namespace mqa {

constexpr int kTcThreads = 192;
constexpr int kTcRows = 128;          // MMA M
constexpr int kTcBufs = 4;            // S and P buffers in tensor memory
constexpr int kTcTmemCols = 512;
constexpr int kTcSCol = 0;                                  // S buffers: kTcBufs x 64 columns
constexpr int kTcPCol = kTcBufs * kTileKeys;                // P buffers: kTcBufs x 32 columns
constexpr int kTcOCol = kTcPCol + kTcBufs * kTileKeys / 2;  // O: d_h columns
constexpr int kTcStageCols = 16;      // columns of O staged per round of the epilogue merge
constexpr int kTcStageStride = kTcStageCols + 1;  // floats per staged row (padded)
constexpr int kTcMergeRows = 4;       // merge scratch rows per warp (merge_split_segment)
__host__ __device__ constexpr int tc_tile_bytes(int D) { return kTileKeys * D * 2; }  // K or V
__host__ __device__ constexpr int tc_k_stages(int D) { return D == 128 ? 5 : 8; }
__host__ __device__ constexpr int tc_v_stages(int D) { return D == 128 ? 6 : 8; }
static_assert(kTcOCol + 128 <= kTcTmemCols, "tensor-memory columns");
static_assert(tc_k_stages(128) >= kTcBufs && tc_k_stages(64) >= kTcBufs,
              "a K tile for every score buffer in flight");

__host__ __device__ constexpr int tc_q_bytes(int D) { return kTcRows * D * 2; }
__host__ __device__ constexpr int tc_barrier_count(int D) {
  return 2 * tc_k_stages(D) + 2 * tc_v_stages(D) + 1 + 3 * kTcBufs + 5;
}
// shared scratch: the epilogue's [128][kTcStageStride] staging, or merge_split_segment's
// 4 x kTcMergeRows rows of comb_row_floats(D)
__host__ __device__ constexpr int tc_scratch_floats(int D) {
  return kTcRows * kTcStageStride > 4 * kTcMergeRows * comb_row_floats(D)
             ? kTcRows * kTcStageStride
             : 4 * kTcMergeRows * comb_row_floats(D);
}
__host__ __device__ constexpr int tc_smem_fixed_bytes(int D) {
  return (tc_k_stages(D) + tc_v_stages(D)) * tc_tile_bytes(D) + tc_q_bytes(D) +
         tc_scratch_floats(D) * 4 + kTcRows * 8 + tc_barrier_count(D) * 8 + 32;
}
// At least 120 KB, so that one CTA fills an SM: two would not both get 512 tensor-memory columns.
__host__ __device__ constexpr size_t tc_smem_bytes(int D) {
  const size_t need = 1024 + static_cast<size_t>(tc_smem_fixed_bytes(D));
  return need > 120 * 1024 ? need : 120 * 1024;
}

struct TcShared {
  SharedLayout base;   // K ring (stages, full, empty), merge scratch (comb_o), cbar, flags, tiles
  uint8_t* vring;      // V ring, after the K ring
  uint64_t* v_full;    // [V stages] a V tile landed (bulk-copy transaction count)
  uint64_t* v_empty;   // [V stages] O += P V of the tile in the stage finished (MMA commit)
  uint8_t* q;          // [D/64][128 rows][128 B], 128-byte swizzle, 1024-aligned
  float2* ml;          // [128] (m_ref, l) of every row at a segment's end
  uint64_t* s_full;    // [kTcBufs] S of tile k is complete (MMA commit), instance k % kTcBufs
  uint64_t* p_full;    // [kTcBufs] P of tile k is in tensor memory (128 softmax threads)
  uint64_t* pv_done;   // [kTcBufs] O += P V of tile k is complete (MMA commit)
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
  t.base.stages = p;   // K ring
  t.vring = p + tc_k_stages(D) * tc_tile_bytes(D);
  p += (tc_k_stages(D) + tc_v_stages(D)) * tc_tile_bytes(D);
  t.q = p;
  p += tc_q_bytes(D);
  t.base.comb_o = reinterpret_cast<float*>(p);
  p += tc_scratch_floats(D) * 4;
  t.ml = reinterpret_cast<float2*>(p);
  t.base.comb_ml = t.ml;  // not used by this kernel's merge path
  p += kTcRows * 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  constexpr int NK = tc_k_stages(D), NV = tc_v_stages(D);
  t.base.full = bars;
  t.base.empty = bars + NK;
  t.v_full = bars + 2 * NK;
  t.v_empty = bars + 2 * NK + NV;
  t.base.cbar = bars + 2 * NK + 2 * NV;
  t.s_full = t.base.cbar + 1;
  t.p_full = t.s_full + kTcBufs;
  t.pv_done = t.p_full + kTcBufs;
  t.q_full = t.pv_done + kTcBufs;
  t.tmem_done = t.q_full + 1;
  t.drain = t.tmem_done + 1;
  t.base.stall = t.drain + 1;
  p += tc_barrier_count(D) * 8;
  t.base.abort = reinterpret_cast<volatile int*>(p);
  t.base.merge = t.base.abort + 1;
  t.tmem_base = reinterpret_cast<uint32_t*>(p + 8);
  return t;
}

// Byte offset of 16-byte chunk c of row r in the swizzled Q tile.
__device__ __forceinline__ uint32_t tc_q_offset(int r, int c) {
  return (c >> 3) * (kTcRows * kSwizzleRowBytes) + r * kSwizzleRowBytes +
         (((c & 7) ^ (r & 7)) << 4);
}

// Q of segment (bi, j) into rows c * GP + h (h < G) of every copy c (128 consumer threads; the
// same thread always writes the same chunks).
template <int D, int GP>
__device__ __forceinline__ void tc_write_q(const DecodeParams& P, const TcShared& sh, int bi,
                                           int j) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int C = kTcRows / GP;
  const uint4* src = reinterpret_cast<const uint4*>(
      P.q + (static_cast<size_t>(bi) * P.h + static_cast<size_t>(j) * P.G) * D);
  for (int e = threadIdx.x; e < P.G * CH; e += 128) {
    const int h = e / CH, c = e - (e / CH) * CH;
    const uint4 v = __ldg(src + e);
#pragma unroll
    for (int cp = 0; cp < C; ++cp)
      *reinterpret_cast<uint4*>(sh.q + tc_q_offset(cp * GP + h, c)) = v;
  }
}

// ---------------------------------------------------------------------------------------------
// MMA issue (one lane of warp 5). Tile k uses K stage k % NK, V stage k % NV and tensor-memory
// buffers k % kTcBufs.
// ---------------------------------------------------------------------------------------------
template <int D>
struct TcMma {
  static constexpr uint32_t kIdescS = umma_idesc_bf16_f32(kTcRows, kTileKeys, false);
  static constexpr uint32_t kIdescO = umma_idesc_bf16_f32(kTcRows, D, true);
  uint32_t kring, vring, q, tmem;

  // S(k) = Q K_k^T: K-steps of 16 along d_h; both operands K-major, 8-row groups 1024 B apart,
  // the second 64-column half of a row 16 KB (Q) or 8 KB (K) further on.
  __device__ __forceinline__ void scores(int k) const {
    const uint32_t kst = kring + (k % tc_k_stages(D)) * tc_tile_bytes(D);
    const uint32_t d_tmem = tmem + kTcSCol + (k % kTcBufs) * kTileKeys;
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
    const uint32_t vst = vring + (k % tc_v_stages(D)) * tc_tile_bytes(D);
    const uint32_t p_tmem = tmem + kTcPCol + (k % kTcBufs) * (kTileKeys / 2);
#pragma unroll
    for (int kk = 0; kk < kTileKeys / 16; ++kk) {
      const uint64_t b = sw128_desc(vst + kk * 16 * kSwizzleRowBytes,
                                    kTileKeys * kSwizzleRowBytes, 1024);
      umma_ts(tmem + kTcOCol, p_tmem + kk * 8, b, kIdescO, (overwrite && kk == 0) ? 0u : 1u);
    }
  }
};

// Barrier instances: tile k uses s_full / p_full / pv_done[k % kTcBufs] at phase k / kTcBufs. No
// waiter can be kTcBufs phases away from the one it asks for (a parity test cannot tell those
// apart): S(k) is issued only after O += P(k - kTcBufs) V finished, which needs P(k - kTcBufs);
// P(k) needs S(k); and the issuer only ever asks for tiles within that window.
//
// The issuer is an event loop: it issues the next tile's scores as soon as that tile's stage has
// landed (and its buffers are free, and, at a segment's start, its Q is in place), and the next
// P V product as soon as that tile's P is ready, whichever comes first. A blocking wait on either
// would hold the other back: a score MMA ahead waits on a bulk copy whose stage only a P V
// product frees. It gives up when nothing has progressed for the wait limit.
template <int D>
__device__ __forceinline__ void tc_issue_loop(const DecodeParams& P, const TcShared& sh,
                                              uint32_t tmem, unsigned long long x0, int ntiles) {
  constexpr int NK = tc_k_stages(D), NV = tc_v_stages(D);
  const SharedLayout& b = sh.base;
  TcMma<D> mma{smem_addr(b.stages), smem_addr(sh.vring), smem_addr(sh.q), tmem};
  TileCursor cur, cs;  // cur: the tile whose P V comes next (k); cs: the next to score (ks)
  cur.start(x0, b.tix);
  cs = cur;
  uint32_t qnext = 0;  // phase of q_full that the next segment start needs
  int k = 0, ks = 0;
  uint64_t last = global_timer_ns();
  for (uint32_t polls = 1; k < ntiles; ++polls) {
    bool progressed = false;
    if (ks < ntiles && ks < k + kTcBufs) {
      const bool need_q = (ks == 0 || cs.tile == 0);
      if ((ks < kTcBufs ||
           mbar_test(&sh.pv_done[ks % kTcBufs], ((ks - kTcBufs) / kTcBufs) & 1)) &&
          mbar_test(&b.full[ks % NK], (ks / NK) & 1) &&  // K tile landed
          (!need_q || mbar_test(sh.q_full, qnext & 1))) {
        if (need_q) ++qnext;
        tc_fence_after_sync();
        mma.scores(ks);
        umma_commit(&sh.s_full[ks % kTcBufs]);
        umma_commit(&b.empty[ks % NK]);  // the K stage is free once the scores are done
        cs.advance(b.tix);
        ++ks;
        progressed = true;
      }
    }
    if (k < ks && mbar_test(&sh.p_full[k % kTcBufs], (k / kTcBufs) & 1) &&
        mbar_test(&sh.v_full[k % NV], (k / NV) & 1)) {
      tc_fence_after_sync();
      mma.values(k, k == 0 || cur.tile == 0);
      umma_commit(&sh.pv_done[k % kTcBufs]);
      umma_commit(&sh.v_empty[k % NV]);
      cur.advance(b.tix);
      ++k;
      progressed = true;
    }
    if (progressed) {
      last = global_timer_ns();
      continue;
    }
    if ((polls & 63u) == 0u) {
      if (*b.abort) return;
      const uint64_t now = global_timer_ns();
      if (now - last > P.timeout_ns) {
        // report what the loop was waiting for
        const int site = ks < k + kTcBufs && ks < ntiles ? kSiteMmaFull : kSiteMmaP;
        give_up(b, site, site == kSiteMmaP ? k : ks);
        return;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Softmax and epilogue (warps 0-3; thread t = row t = tensor-memory lane t). Returns false if a
// wait timed out (the wait has recorded itself).
// ---------------------------------------------------------------------------------------------
template <int D, int GP>
__device__ __forceinline__ bool tc_softmax_loop(const DecodeParams& P, const TcShared& sh,
                                                uint32_t tmem, unsigned long long x0, int ntiles,
                                                unsigned long long W) {
  constexpr int C = kTcRows / GP;          // copies of the group
  constexpr int OWN = kTileKeys / C;       // keys of a tile each copy owns
  constexpr int KW = OWN < 16 ? 16 : OWN;  // keys a warp loads (the copies it holds)
  const SharedLayout& b = sh.base;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = P.G;
  const int copy = tid / GP, head = tid - copy * GP;
  const int own0 = copy * OWN;                  // first key of this row's range
  const int kw0 = ((32 * warp) / GP) * OWN;     // first key this warp loads
  const bool second_half = (own0 - kw0) != 0;   // only when KW = 2 * OWN (GP = 16)
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  uint32_t cphase = 0;

  // the P buffers start at zero: each row later writes only the columns of its own keys
  {
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
    for (int bf = 0; bf < kTcBufs; ++bf)
      tmem_st_32x32b_x32(tmem + lane_base + kTcPCol + bf * (kTileKeys / 2), z);
    tmem_wait_st();
  }
  TileCursor cur;
  cur.start(x0, b.tix);
  tc_write_q<D, GP>(P, sh, cur.bi, cur.j);
  fence_proxy_async_smem();
  mbar_arrive(sh.q_full);

  float m_ref = -INFINITY, l = 0.f;
  int L = 0;
  bool began_at_zero = false;
  if (P.debug_stall) {
    const bool ok = mbar_wait_bounded(b.stall, 0, P.timeout_ns, b.abort);
    if (!ok && !*b.abort) give_up(b, kSiteStall, 0);
    if (!__all_sync(0xffffffffu, ok)) return false;
  }
  for (int k = 0; k < ntiles; ++k) {
    const bool first = (k == 0 || cur.tile == 0);
    if (first) {
      L = __ldg(P.seq_lens + cur.bi);
      began_at_zero = (cur.tile == 0);
      m_ref = -INFINITY;
      l = 0.f;
    }
    const int valid = min(L - cur.tile * kTileKeys, kTileKeys);  // >= 1
    const int bf = k % kTcBufs;
    bool ok = mbar_wait_bounded(&sh.s_full[bf], (k / kTcBufs) & 1, P.timeout_ns, b.abort);
    if (!ok && !*b.abort) give_up(b, kSiteSoftmaxS, k);
    if (!__all_sync(0xffffffffu, ok)) return false;
    tc_fence_after_sync();

    // this row's scores, scaled to log2 units; keys at or past the length are -inf
    float s[OWN];
    {
      uint32_t r[KW];
      const uint32_t taddr = tmem + lane_base + kTcSCol + bf * kTileKeys + kw0;
      if constexpr (KW == 16) tmem_ld_32x32b_x16(taddr, r);
      else tmem_ld_32x32b_x32(taddr, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < OWN; ++i) {
        const uint32_t raw = (KW == OWN) ? r[i] : (second_half ? r[i + (KW - OWN)] : r[i]);
        s[i] = own0 + i < valid ? __uint_as_float(raw) * P.scale_log2 : -INFINITY;
      }
    }
    float mx = s[0];
#pragma unroll
    for (int i = 1; i < OWN; ++i) mx = fmaxf(mx, s[i]);
    float alpha = 1.f;
    bool raise = false;
    if (first) {
      m_ref = mx;                     // -inf when this copy has no valid key in the tile
    } else if (mx > m_ref + kLazyLog2) {
      raise = true;
      alpha = fast_exp2(m_ref - mx);  // 0 when m_ref is -inf
      m_ref = mx;
      l *= alpha;
    }
    if (__any_sync(0xffffffffu, raise)) {
      // O must hold P V of the previous tile before its rows are rescaled
      const int kp = k - 1;
      ok = mbar_wait_bounded(&sh.pv_done[kp % kTcBufs], (kp / kTcBufs) & 1, P.timeout_ns,
                             b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteSoftmaxPv, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTcOCol + c, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_32x32b_x32(tmem + lane_base + kTcOCol + c, o);
      }
      tmem_wait_st();
    }
    // probabilities, rounded to bf16 once: the same values feed P V and the running sum
    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
    uint32_t pk[KW / 2];
    float ps = 0.f;
#pragma unroll
    for (int i = 0; i < OWN / 2; ++i) {
      const uint32_t v =
          pack_bf16x2(fast_exp2(s[2 * i] - m_use), fast_exp2(s[2 * i + 1] - m_use));
      ps += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
      if constexpr (KW == OWN) {
        pk[i] = v;
      } else {
        pk[i] = second_half ? 0u : v;
        pk[i + OWN / 2] = second_half ? v : 0u;
      }
    }
    l += ps;
    {
      const uint32_t taddr = tmem + lane_base + kTcPCol + bf * (kTileKeys / 2) + kw0 / 2;
      if constexpr (KW == 16) tmem_st_32x32b_x8(taddr, pk);
      else tmem_st_32x32b_x16(taddr, pk);
    }
    tmem_wait_st();

    if (valid < kTileKeys) {
      // V rows at or beyond the length may hold anything (NaN included), and 0 * NaN = NaN in
      // the MMA: zero them. The stage's full barrier is complete (the scores read its K half);
      // waiting on it orders the bulk copy's writes before these.
      constexpr int NV = tc_v_stages(D);
      const int st = k % NV;
      ok = mbar_wait_bounded(&sh.v_full[st], (k / NV) & 1, P.timeout_ns, b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteSoftmaxFull, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      uint8_t* vst = sh.vring + st * tc_tile_bytes(D);
      constexpr int CH = D / 8;
      for (int e = tid; e < (kTileKeys - valid) * CH; e += 128) {
        const int key = valid + e / CH, c = e - (e / CH) * CH;
        *reinterpret_cast<uint4*>(vst + (c >> 3) * (kTileKeys * kSwizzleRowBytes) +
                                  key * kSwizzleRowBytes + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    mbar_arrive(&sh.p_full[bf]);

    TileCursor nxt = cur;
    nxt.advance(b.tix);
    const bool has_next = k + 1 < ntiles;
    if (has_next && nxt.tile == 0) {
      // the next tile starts a segment; every score MMA of this one (S(k) last) has finished
      tc_write_q<D, GP>(P, sh, nxt.bi, nxt.j);
      fence_proxy_async_smem();
      mbar_arrive(sh.q_full);
    }

    const bool seg_end = (cur.tile == cur.nt - 1);
    if (seg_end || !has_next) {
      ok = mbar_wait_bounded(&sh.pv_done[bf], (k / kTcBufs) & 1, P.timeout_ns, b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteEpiloguePv, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after_sync();
      const bool complete = began_at_zero && seg_end;
      const int seg = cur.bi * P.g + cur.j;
      const size_t slot = static_cast<size_t>(blockIdx.x) + seg;
      // merge the C copies of every head: M = max_c m_c, L = sum_c 2^(m_c - M) l_c, and each
      // row's weight 2^(m_c - M) (divided by L for the final output)
      sh.ml[tid] = make_float2(m_ref, l);
      if (!consumer_sync(b, cphase, P.timeout_ns)) {
        if (!*b.abort) give_up(b, kSiteConsumerSync, k);
        return false;
      }
      float M = -INFINITY, Lsum = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) M = fmaxf(M, sh.ml[c * GP + head].x);
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const float2 v = sh.ml[c * GP + head];
        Lsum += v.y == 0.f ? 0.f : fast_exp2(v.x - M) * v.y;
      }
      const float wr = (l == 0.f ? 0.f : fast_exp2(m_ref - M)) * (complete ? 1.f / Lsum : 1.f);
      if (!complete && tid < G) P.part_ml[slot * G + tid] = make_float2(M, Lsum);
      float* stg = b.comb_o;  // [128][kTcStageStride]
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += kTcStageCols) {
        uint32_t o[kTcStageCols];
        tmem_ld_32x32b_x16(tmem + lane_base + kTcOCol + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kTcStageCols; ++i)
          stg[tid * kTcStageStride + i] = __uint_as_float(o[i]) * wr;
        if (!consumer_sync(b, cphase, P.timeout_ns)) {
          if (!*b.abort) give_up(b, kSiteConsumerSync, k);
          return false;
        }
        for (int idx = tid; idx < G * kTcStageCols; idx += 128) {
          const int hh = idx / kTcStageCols, col = idx % kTcStageCols;
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < C; ++c) acc += stg[(c * GP + hh) * kTcStageStride + col];
          if (complete)
            P.out[(static_cast<size_t>(cur.bi) * P.h + static_cast<size_t>(cur.j) * G + hh) * D +
                  c0 + col] = __float2bfloat16_rn(acc);
          else
            P.part_o[(slot * G + hh) * D + c0 + col] = acc;
        }
        if (!consumer_sync(b, cphase, P.timeout_ns)) {
          if (!*b.abort) give_up(b, kSiteConsumerSync, k);
          return false;
        }
      }
      if (!complete) {
        __threadfence();  // this CTA's partial is visible before it is counted
        if (!consumer_sync(b, cphase, P.timeout_ns) ||
            !finish_split_segment<D, 4, kTcMergeRows>(P, b, cphase, cur, W)) {
          if (!*b.abort) give_up(b, kSiteConsumerSync, k);
          return false;
        }
      }
    }
    cur = nxt;
  }
  return true;
}

// ---------------------------------------------------------------------------------------------
// Producer (warp 4): K and V tiles into their rings with bulk tensor copies (lane 0), each as soon
// as its stage is free, V never ahead of K; for the fused append, the tile's new K and V rows are
// written first (whole warp), as in produce_tiles. Gives up when nothing progressed for the wait
// limit; then waits (bounded) for its copies in flight.
// ---------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void tc_produce_tiles(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                 const DecodeParams& P, const TcShared& sh,
                                                 unsigned long long x0, int ntiles, int lane) {
  constexpr uint32_t kTile = tc_tile_bytes(D);
  constexpr int NK = tc_k_stages(D), NV = tc_v_stages(D);
  const SharedLayout& b = sh.base;
  const bool fused = P.pos != nullptr;
  if (!fused && lane != 0) return;
  if (lane == 0) {
    prefetch_tensor_map(tm_k);
    prefetch_tensor_map(tm_v);
  }
  const uint64_t policy = l2_policy_evict_first();
  TileCursor ck, cv;
  ck.start(x0, b.tix);
  cv = ck;
  int kk = 0, kv = 0;
  int row_bi = -1, row_p = -1;
  uint64_t last = global_timer_ns();
  for (uint32_t polls = 1; kv < ntiles; ++polls) {
    int act = 0;  // 1: issue K tile kk, 2: issue V tile kv
    if (lane == 0) {
      if (kk < ntiles && mbar_test(&b.empty[kk % NK], ((kk / NK) & 1) ^ 1)) act = 1;
      else if (kv < kk && mbar_test(&sh.v_empty[kv % NV], ((kv / NV) & 1) ^ 1)) act = 2;
    }
    if (fused) act = __shfl_sync(0xffffffffu, act, 0);
    if (act == 1) {
      if (fused) {
        if (ck.bi != row_bi) {
          row_bi = ck.bi;
          const int p = __ldg(P.pos + ck.bi);
          row_p = (p >= 0 && p < P.n_max) ? p : -1;
        }
        if (row_p >= 0 && row_p / kTileKeys == ck.tile) {
          write_new_row<D, 2>(P, ck.bi, ck.j, 0, row_p, lane);
          fence_proxy_async_global();  // each writer orders its stores before the async proxy...
          __syncwarp();                // ...and lane 0 copies the tile after every writer
        }
      }
      if (lane == 0) {
        const int st = kk % NK;
        mbar_arrive_expect_tx(&b.full[st], kTile);
        uint8_t* dst = b.stages + st * kTile;
#pragma unroll
        for (int half = 0; half < D / 64; ++half)
          tma_load_3d(dst + half * kTileKeys * kSwizzleRowBytes, tm_k, &b.full[st], half * 64,
                      ck.tile * kTileKeys, ck.bi * P.g + ck.j, policy);
      }
      ck.advance(b.tix);
      ++kk;
    } else if (act == 2) {
      if (lane == 0) {
        const int st = kv % NV;
        mbar_arrive_expect_tx(&sh.v_full[st], kTile);
        uint8_t* dst = sh.vring + st * kTile;
#pragma unroll
        for (int half = 0; half < D / 64; ++half)
          tma_load_3d(dst + half * kTileKeys * kSwizzleRowBytes, tm_v, &sh.v_full[st], half * 64,
                      cv.tile * kTileKeys, cv.bi * P.g + cv.j, policy);
      }
      cv.advance(b.tix);
      ++kv;
    }
    if (act != 0) {
      if (lane == 0) last = global_timer_ns();
      continue;
    }
    int stop = 0;
    if (lane == 0 && (polls & 63u) == 0u) {
      if (*b.abort) {
        stop = 1;
      } else if (global_timer_ns() - last > P.timeout_ns) {
        give_up(b, kSiteProducerEmpty, kk);
        stop = 1;
      }
    }
    if (fused) stop = __shfl_sync(0xffffffffu, stop, 0);
    if (stop) break;
  }
  if (lane != 0) return;
  // let the copies still in flight land before the CTA may exit (bounded; no-op normally)
  const volatile int never = 0;
  for (int i = kk > NK ? kk - NK : 0; i < kk; ++i)
    mbar_wait_bounded(&b.full[i % NK], (i / NK) & 1, P.drain_ns, &never);
  for (int i = kv > NV ? kv - NV : 0; i < kv; ++i)
    mbar_wait_bounded(&sh.v_full[i % NV], (i / NV) & 1, P.drain_ns, &never);
}

// ---------------------------------------------------------------------------------------------
// The kernel. GP = the group size padded to 16, 32 or 64.
// ---------------------------------------------------------------------------------------------
template <int D, int GP>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v, const DecodeParams P) {
  static_assert(GP == 16 || GP == 32 || GP == 64, "padded group size");
  extern __shared__ uint8_t smem_raw[];
  TcShared sh = carve_tc_shared<D>(smem_raw);
  SharedLayout& b = sh.base;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (warp == 5) {
    tmem_alloc(sh.tmem_base, kTcTmemCols);
    tmem_relinquish_alloc_permit();
  }
  __shared__ uint32_t chunk_tiles[kTcThreads + 1];
  if (tid == 0) {
    *b.abort = 0;
    *b.merge = 0;
    for (int st = 0; st < tc_k_stages(D); ++st) {
      mbar_init(&b.full[st], 1);       // K ring
      mbar_init(&b.empty[st], 1);      // one MMA commit frees a stage
    }
    for (int st = 0; st < tc_v_stages(D); ++st) {
      mbar_init(&sh.v_full[st], 1);    // V ring
      mbar_init(&sh.v_empty[st], 1);
    }
    mbar_init(b.cbar, 128);
    for (int i = 0; i < kTcBufs; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 128);
      mbar_init(&sh.pv_done[i], 1);
    }
    mbar_init(sh.q_full, 128);
    mbar_init(sh.tmem_done, 128);
    mbar_init(sh.drain, 1);
    mbar_init(b.stall, 1);
    fence_barrier_init();
  }
  // rows of heads G .. GP-1 of every copy stay zero for the whole launch; the CTA-wide barrier
  // below orders these writes before any Q row is written or read
  {
    constexpr int CH = D / 8;
    const int per_copy = (GP - P.G) * CH;
    for (int e = tid; e < (kTcRows / GP) * per_copy; e += kTcThreads) {
      const int cp = e / per_copy, rem = e - cp * per_copy;
      const int r = cp * GP + P.G + rem / CH, c = rem % CH;
      *reinterpret_cast<uint4*>(sh.q + tc_q_offset(r, c)) = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before_sync();
  build_tile_prefix<kTcThreads>(P, b, chunk_tiles);  // ends with a CTA-wide barrier
  tc_fence_after_sync();
  const uint32_t tmem = *sh.tmem_base;

  zero_invalid_sequences<D>(P, kTcThreads);
  if (P.pos != nullptr) append_uncovered_rows<D, 2>(P, kTcThreads);

  const unsigned long long W = b.tix.total();
  const unsigned long long x0 = W * blockIdx.x / P.num_ctas;
  const unsigned long long x1 = W * (blockIdx.x + 1) / P.num_ctas;
  if (x0 >= x1) {
    if (warp == 5) tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  const int ntiles = static_cast<int>(x1 - x0);

  if (warp == 4) {
    tc_produce_tiles<D>(&tm_k, &tm_v, P, sh, x0, ntiles, lane);
    return;
  }
  if (warp == 5) {
    const volatile int never = 0;
    if (lane == 0) {
      tc_issue_loop<D>(P, sh, tmem, x0, ntiles);
      // every MMA issued has finished, and the softmax warps are done, before the columns go
      umma_commit(sh.drain);
      if (!mbar_wait_bounded(sh.drain, 0, P.drain_ns, &never)) give_up(b, kSiteDrain, ntiles);
      if (!mbar_wait_bounded(sh.tmem_done, 0, P.drain_ns + 2 * P.timeout_ns, &never))
        give_up(b, kSiteTmemDone, ntiles);
    }
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTcTmemCols);
    return;
  }
  // warps 0-3
  tc_softmax_loop<D, GP>(P, sh, tmem, x0, ntiles, W);  // a timed-out wait has recorded itself
  tc_fence_before_sync();
  mbar_arrive(sh.tmem_done);
}

}  // namespace mqa
