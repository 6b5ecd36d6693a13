// prefill_attention_tc.cuh -- causal grouped attention of many new tokens per sequence (a
// prefill-sized T) on the 5th-generation tensor cores (tcgen05.mma, accumulators in tensor
// memory) for sm_103a.
//
// Definition ("分组查询注意力（GQA）与多查询注意力（MQA）深度实战", ybb.press, §八 with the causal mask
// of §十 item 10): the T new tokens of sequence bi sit at cache rows L - T .. L - 1 (L =
// seq_lens[bi]); token t attends the first L - T + 1 + t rows, and query head i of token t reads
// KV head j = i / Gh (Gh = h / g):
//     out[bi][t][i] = sum_{s < L-T+1+t} softmax_s(scale q[bi][t][i] . K[bi][j][s]) V[bi][j][s].
// This is the several-token decode of decode_attention.cuh with T large enough that the rows of a
// KV head (T * Gh of them) no longer fit one tile of heads: here the score and value products
// are real matrix products of 128 query rows by 64 keys, the shape the tensor cores are made for.
//
// Work. The rows of segment (bi, j) are r = t * Gh + hh (hh < Gh), T * Gh of them, cut into
// blocks of 128. A unit is one block: its 128 rows and the key tiles [0, nt) its last row sees
// (nt = ceil(lim / 64), lim = L - T + 1 + t_last). Units are numbered u = (bi * g + j) * NB + rb
// (NB blocks per segment) and CTA c of P takes units c, c + P, c + 2P, ...; a unit is finished
// inside its CTA, so there are no partial states. The units of one segment are consecutive, so
// the CTAs that read a segment's K and V run at about the same time and share them through L2.
//
// Inside a CTA (192 threads, the roles of the decode tcgen05 kernel; two CTAs per SM): warps 0-3
// own one row each per thread (thread t = row t of the block = tensor-memory lane t): they write
// the unit's Q into shared memory, run the online softmax with the row's own causal limit, and
// write the output row; warp 4 streams the K and V tiles with bulk tensor copies into separate
// rings; one lane of warp 5 issues the MMAs from an event loop and warp 5 owns the tensor memory.
//
//   S = Q K^T      M = 128 rows, N = 64 keys, K = d_h; A = Q, B = the K tile (shared memory,
//                  128-byte swizzle); S in tensor memory, fp32, kPfBufs buffers
//   softmax        thread r loads its 64 scores, masks the keys past its limit, and writes its
//                  bf16 probabilities over the first 32 columns of its row of that S buffer
//   O += P V       M = 128, N = d_h, K = 64 keys; A = P (tensor memory), B = the V tile
//                  (N-major); O in tensor memory, fp32
//
// The softmax reference is lazy (raised, and O rescaled, only when a row's maximum grows by more
// than kLazyLog2), the weights are rounded to bf16 once and the running sum adds exactly those
// rounded weights, as on the decode paths. The new rows are appended beforehand by a separate
// launch (the T rows of a sequence are read by every unit of its segments).
//
// Every wait is bounded in time; on expiry the kernel records the wait, latches MQA_ERR_TIMEOUT,
// and warp 5 waits (bounded) for its MMAs and for the softmax warps before it frees the tensor
// memory.
#pragma once

#include "decode_attention_tc.cuh"

namespace mqa {

constexpr int kPfRows = kTcRows;  // rows per unit (MMA M)
constexpr int kMaxPrefillRows = 1 << 22;  // largest T * h / g served

// Two CTAs per SM, so that every SM sub-partition runs two softmax warps whose per-tile chains
// hide each other's latency: each CTA takes half the tensor memory and under half the shared
// memory. Tensor memory (256 columns per CTA): kPfBufs S buffers of 64 columns, and O; the bf16
// probabilities P of a tile go back into the first 32 columns of its own S buffer once the
// scores are in registers (an S buffer is reused only after the P V that read its P finished).
constexpr int kPfCtasPerSm = 2;
constexpr int kPfBufs = 2;
constexpr int kPfTmemCols = 256;
constexpr int kPfSCol = 0;                       // S (then P) buffers: kPfBufs x 64 columns
constexpr int kPfOCol = kPfBufs * kTileKeys;     // O: d_h columns
static_assert(kPfOCol + 128 <= kPfTmemCols, "tensor-memory columns");
__host__ __device__ constexpr int pf_k_stages(int D) { return D == 128 ? 2 : 4; }
__host__ __device__ constexpr int pf_v_stages(int D) { return D == 128 ? 2 : 4; }
__host__ __device__ constexpr int pf_barrier_count(int D) {
  return 2 * pf_k_stages(D) + 2 * pf_v_stages(D) + 1 + 3 * kPfBufs + 4;
}
__host__ __device__ constexpr size_t pf_smem_bytes(int D) {
  return 1024 + static_cast<size_t>((pf_k_stages(D) + pf_v_stages(D)) * tc_tile_bytes(D) +
                                    tc_q_bytes(D) + pf_barrier_count(D) * 8 + 32);
}
static_assert(pf_smem_bytes(128) <= 110 * 1024 && pf_smem_bytes(64) <= 110 * 1024,
              "two CTAs per SM");

// The prefill kernel's shared memory, in the decode tcgen05 kernel's struct (the bounded waits
// and give_up use its fields): the K ring, the V ring, Q, and the barriers.
template <int D>
__device__ __forceinline__ TcShared carve_pf_shared(uint8_t* raw) {
  TcShared t = {};
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  constexpr int NK = pf_k_stages(D), NV = pf_v_stages(D);
  t.base.stages = p;  // K ring
  t.vring = p + NK * tc_tile_bytes(D);
  p += (NK + NV) * tc_tile_bytes(D);
  t.q = p;
  p += tc_q_bytes(D);
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  t.base.full = bars;
  t.base.empty = bars + NK;
  t.v_full = bars + 2 * NK;
  t.v_empty = bars + 2 * NK + NV;
  t.s_full = bars + 2 * NK + 2 * NV;
  t.p_full = t.s_full + kPfBufs;
  t.pv_done = t.p_full + kPfBufs;
  t.q_full = t.pv_done + kPfBufs;
  t.tmem_done = t.q_full + 1;
  t.drain = t.tmem_done + 1;
  t.base.stall = t.drain + 1;
  t.base.cbar = t.base.stall + 1;  // unused
  p += pf_barrier_count(D) * 8;
  t.base.abort = reinterpret_cast<volatile int*>(p);
  t.base.merge = t.base.abort + 1;
  t.tmem_base = reinterpret_cast<uint32_t*>(p + 8);
  return t;
}

// MMA issue for tile k: S into buffer k % kPfBufs; O += P V with P from the first 32 columns of
// that buffer. The descriptors are those of the decode tcgen05 kernel's scores and values.
template <int D>
struct PfMma {
  static constexpr uint32_t kIdescS = umma_idesc_bf16_f32(kTcRows, kTileKeys, false);
  static constexpr uint32_t kIdescO = umma_idesc_bf16_f32(kTcRows, D, true);
  uint32_t kring, vring, q, tmem;
  __device__ __forceinline__ void scores(int k) const {
    const uint32_t kst = kring + (k % pf_k_stages(D)) * tc_tile_bytes(D);
    const uint32_t d_tmem = tmem + kPfSCol + (k % kPfBufs) * kTileKeys;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk & 3) * 32;
      const uint64_t a = sw128_desc(q + (kk >> 2) * (kTcRows * kSwizzleRowBytes) + off, 0, 1024);
      const uint64_t bd = sw128_desc(kst + (kk >> 2) * (kTileKeys * kSwizzleRowBytes) + off, 0,
                                     1024);
      umma_ss(d_tmem, a, bd, kIdescS, kk > 0 ? 1u : 0u);
    }
  }
  __device__ __forceinline__ void values(int k, bool overwrite) const {
    const uint32_t vst = vring + (k % pf_v_stages(D)) * tc_tile_bytes(D);
    const uint32_t p_tmem = tmem + kPfSCol + (k % kPfBufs) * kTileKeys;
#pragma unroll
    for (int kk = 0; kk < kTileKeys / 16; ++kk) {
      const uint64_t bd = sw128_desc(vst + kk * 16 * kSwizzleRowBytes,
                                     kTileKeys * kSwizzleRowBytes, 1024);
      umma_ts(tmem + kPfOCol, p_tmem + kk * 8, bd, kIdescO, (overwrite && kk == 0) ? 0u : 1u);
    }
  }
};

// Units of the launch: NB blocks of 128 rows per segment, b * g segments.
__device__ __forceinline__ long long pf_blocks(const DecodeParams& P) {
  return (static_cast<long long>(P.G) + kPfRows - 1) / kPfRows;
}
__device__ __forceinline__ long long pf_units(const DecodeParams& P) {
  return static_cast<long long>(P.b) * P.g * pf_blocks(P);
}

// Walks a CTA's units and their key tiles, in the order every role of the CTA uses.
struct PfCursor {
  long long u;  // current unit (>= pf_units when done)
  int bi, j, rb;
  int tile, nt;  // current key tile of the unit, and the unit's tile count
  int L;         // length of sequence bi

  // Unit u's sequence, head and block, and its tile count (0 when the sequence's length is out
  // of range: such sequences get a zero output elsewhere).
  __device__ __forceinline__ void setup(const DecodeParams& P) {
    const long long NB = pf_blocks(P);
    const long long seg = u / NB;
    rb = static_cast<int>(u - seg * NB);
    bi = static_cast<int>(seg / P.g);
    j = static_cast<int>(seg - static_cast<long long>(bi) * P.g);
    L = __ldg(P.seq_lens + bi);
    tile = 0;
    if (L < P.T || L > P.n_max) {
      nt = 0;
      return;
    }
    const int r_last = min(rb * kPfRows + kPfRows, P.G) - 1;
    const int lim = L - P.T + 1 + r_last / P.Gh;  // keys the block's last row sees (>= 1)
    nt = (lim + kTileKeys - 1) / kTileKeys;
  }
  __device__ __forceinline__ void skip_empty(const DecodeParams& P, long long U) {
    while (u < U) {
      setup(P);
      if (nt > 0) return;
      u += P.num_ctas;
    }
  }
  __device__ __forceinline__ void start(const DecodeParams& P, long long U) {
    u = blockIdx.x;
    skip_empty(P, U);
  }
  __device__ __forceinline__ void advance(const DecodeParams& P, long long U) {
    if (++tile < nt) return;
    u += P.num_ctas;
    skip_empty(P, U);
  }
  __device__ __forceinline__ bool done(long long U) const { return u >= U; }
};

// Q of the unit at `c` into the Q tile (thread t writes row t; rows past the segment's T * Gh
// rows are zero).
template <int D>
__device__ __forceinline__ void pf_write_q(const DecodeParams& P, const TcShared& sh,
                                           const PfCursor& c) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int r = c.rb * kPfRows + static_cast<int>(threadIdx.x);
  if (r < P.G) {
    const int t = r / P.Gh, hh = r - t * P.Gh;
    const uint4* src = reinterpret_cast<const uint4*>(
        P.q + ((static_cast<size_t>(c.bi) * P.T + t) * P.h + static_cast<size_t>(c.j) * P.Gh +
               hh) * D);
#pragma unroll
    for (int ch = 0; ch < CH; ++ch)
      *reinterpret_cast<uint4*>(sh.q + tc_q_offset(threadIdx.x, ch)) = __ldg(src + ch);
  } else {
#pragma unroll
    for (int ch = 0; ch < CH; ++ch)
      *reinterpret_cast<uint4*>(sh.q + tc_q_offset(threadIdx.x, ch)) = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------------------------
// MMA issue (one lane of warp 5): the event loop of the decode tcgen05 kernel over the units'
// tiles. Tile k (counted over the CTA's units) uses K stage k % NK, V stage k % NV and the
// tensor-memory buffers k % kPfBufs at phase k / kPfBufs; the S MMAs of a unit's first tile wait
// for its Q (q_full, one phase per unit).
// ---------------------------------------------------------------------------------------------
// Returns the number of tiles whose score MMAs it issued.
template <int D>
__device__ __forceinline__ int pf_issue_loop(const DecodeParams& P, const TcShared& sh,
                                             uint32_t tmem, long long U) {
  constexpr int NK = pf_k_stages(D), NV = pf_v_stages(D);
  const SharedLayout& b = sh.base;
  PfMma<D> mma{smem_addr(b.stages), smem_addr(sh.vring), smem_addr(sh.q), tmem};
  PfCursor cur, cs;  // cur: the tile whose P V comes next (k); cs: the next to score (ks)
  cur.start(P, U);
  cs = cur;
  uint32_t qnext = 0;
  int k = 0, ks = 0;
  uint64_t last = global_timer_ns();
  for (uint32_t polls = 1; !cur.done(U); ++polls) {
    bool progressed = false;
    if (!cs.done(U) && ks < k + kPfBufs) {
      const bool need_q = (cs.tile == 0);
      if ((ks < kPfBufs ||
           mbar_test(&sh.pv_done[ks % kPfBufs], ((ks - kPfBufs) / kPfBufs) & 1)) &&
          mbar_test(&b.full[ks % NK], (ks / NK) & 1) &&
          (!need_q || mbar_test(sh.q_full, qnext & 1))) {
        if (need_q) ++qnext;
        tc_fence_after_sync();
        mma.scores(ks);
        umma_commit(&sh.s_full[ks % kPfBufs]);
        umma_commit(&b.empty[ks % NK]);
        cs.advance(P, U);
        ++ks;
        progressed = true;
      }
    }
    if (k < ks && mbar_test(&sh.p_full[k % kPfBufs], (k / kPfBufs) & 1) &&
        mbar_test(&sh.v_full[k % NV], (k / NV) & 1)) {
      tc_fence_after_sync();
      mma.values(k, cur.tile == 0);
      umma_commit(&sh.pv_done[k % kPfBufs]);
      umma_commit(&sh.v_empty[k % NV]);
      cur.advance(P, U);
      ++k;
      progressed = true;
    }
    if (progressed) {
      last = global_timer_ns();
      continue;
    }
    if ((polls & 63u) == 0u) {
      if (*b.abort) return ks;
      if (global_timer_ns() - last > P.timeout_ns) {
        const bool scoring = !cs.done(U) && ks < k + kPfBufs;
        give_up(b, scoring ? kSiteMmaFull : kSiteMmaP, scoring ? ks : k);
        return ks;
      }
    }
  }
  return ks;
}

// ---------------------------------------------------------------------------------------------
// Producer (warp 4, lane 0): K and V tiles of the CTA's units into their rings as their stages
// free up, V never ahead of K. Gives up when nothing progressed for the wait limit, then waits
// (bounded) for its copies in flight.
// ---------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void pf_produce_tiles(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                 const DecodeParams& P, const TcShared& sh,
                                                 long long U) {
  constexpr uint32_t kTile = tc_tile_bytes(D);
  constexpr int NK = pf_k_stages(D), NV = pf_v_stages(D);
  const SharedLayout& b = sh.base;
  prefetch_tensor_map(tm_k);
  prefetch_tensor_map(tm_v);
  // K and V tiles are read by every unit of a segment: keep them in L2 normally
  PfCursor ck, cv;
  ck.start(P, U);
  cv = ck;
  int kk = 0, kv = 0;
  uint64_t last = global_timer_ns();
  for (uint32_t polls = 1; !cv.done(U); ++polls) {
    bool acted = false;
    if (!ck.done(U) && mbar_test(&b.empty[kk % NK], ((kk / NK) & 1) ^ 1)) {
      const int st = kk % NK;
      mbar_arrive_expect_tx(&b.full[st], kTile);
      uint8_t* dst = b.stages + st * kTile;
#pragma unroll
      for (int half = 0; half < D / 64; ++half)
        tma_load_3d_nohint(dst + half * kTileKeys * kSwizzleRowBytes, tm_k, &b.full[st],
                           half * 64, ck.tile * kTileKeys, ck.bi * P.g + ck.j);
      ck.advance(P, U);
      ++kk;
      acted = true;
    } else if (kv < kk && mbar_test(&sh.v_empty[kv % NV], ((kv / NV) & 1) ^ 1)) {
      const int st = kv % NV;
      mbar_arrive_expect_tx(&sh.v_full[st], kTile);
      uint8_t* dst = sh.vring + st * kTile;
#pragma unroll
      for (int half = 0; half < D / 64; ++half)
        tma_load_3d_nohint(dst + half * kTileKeys * kSwizzleRowBytes, tm_v, &sh.v_full[st],
                           half * 64, cv.tile * kTileKeys, cv.bi * P.g + cv.j);
      cv.advance(P, U);
      ++kv;
      acted = true;
    }
    if (acted) {
      last = global_timer_ns();
      continue;
    }
    if ((polls & 63u) == 0u) {
      if (*b.abort) break;
      if (global_timer_ns() - last > P.timeout_ns) {
        give_up(b, kSiteProducerEmpty, kk);
        break;
      }
    }
  }
  // let the copies still in flight land before the CTA may exit (bounded; no-op normally)
  const volatile int never = 0;
  for (int i = kk > NK ? kk - NK : 0; i < kk; ++i)
    mbar_wait_bounded(&b.full[i % NK], (i / NK) & 1, P.drain_ns, &never);
  for (int i = kv > NV ? kv - NV : 0; i < kv; ++i)
    mbar_wait_bounded(&sh.v_full[i % NV], (i / NV) & 1, P.drain_ns, &never);
}

// ---------------------------------------------------------------------------------------------
// Softmax and epilogue (warps 0-3; thread t = row t of the unit = tensor-memory lane t). Returns
// false if a wait timed out (the wait has recorded itself).
// ---------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ bool pf_softmax_loop(const DecodeParams& P, const TcShared& sh,
                                                uint32_t tmem, long long U) {
  constexpr int NV = pf_v_stages(D);
  const SharedLayout& b = sh.base;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  PfCursor cur;
  cur.start(P, U);
  if (cur.done(U)) return true;
  pf_write_q<D>(P, sh, cur);
  fence_proxy_async_smem();
  mbar_arrive(sh.q_full);

  if (P.debug_stall == 1) {
    const bool ok = mbar_wait_bounded(b.stall, 0, P.timeout_ns, b.abort);
    if (!ok && !*b.abort) give_up(b, kSiteStall, 0);
    if (!__all_sync(0xffffffffu, ok)) return false;
  }
  float m_ref = -INFINITY, l = 0.f;
  int lim = 0;      // keys this row sees (0 for a padding row)
  int t_row = 0, hh = 0;
  for (int k = 0; !cur.done(U); ++k) {
    if (cur.tile == 0) {
      const int r = cur.rb * kPfRows + tid;
      if (r < P.G) {
        t_row = r / P.Gh;
        hh = r - t_row * P.Gh;
        lim = cur.L - P.T + 1 + t_row;
      } else {
        lim = 0;
      }
      m_ref = -INFINITY;
      l = 0.f;
    }
    const int bf = k % kPfBufs;
    bool ok = mbar_wait_bounded(&sh.s_full[bf], (k / kPfBufs) & 1, P.timeout_ns, b.abort);
    if (!ok && !*b.abort) give_up(b, kSiteSoftmaxS, k);
    if (!__all_sync(0xffffffffu, ok)) return false;
    tc_fence_after_sync();

    // this row's 64 raw scores; the first nvis keys are visible to the row (its causal limit
    // and the sequence's end), the rest are masked. Scaled scores are s * sc (log2 units); the
    // row's largest scaled score comes from the largest raw score (or the smallest, for a
    // negative scale), so the scale is applied once per key, inside the exponential's FFMA.
    const int key0 = cur.tile * kTileKeys;
    const int nvis = min(max(lim - key0, 0), kTileKeys);
    const float sc = P.scale_log2;
    const bool all_visible = __all_sync(0xffffffffu, nvis == kTileKeys);
    float s[kTileKeys];
    {
      uint32_t r0[32], r1[32];
      const uint32_t taddr = tmem + lane_base + kPfSCol + bf * kTileKeys;
      tmem_ld_32x32b_x32(taddr, r0);
      tmem_ld_32x32b_x32(taddr + 32, r1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(r0[i]);
        s[32 + i] = __uint_as_float(r1[i]);
      }
    }
    float ext;
    if (sc >= 0.f) {
      ext = -INFINITY;
      if (all_visible) {
#pragma unroll
        for (int i = 0; i < kTileKeys; ++i) ext = fmaxf(ext, s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kTileKeys; ++i) ext = i < nvis ? fmaxf(ext, s[i]) : ext;
      }
    } else {
      ext = INFINITY;
      if (all_visible) {
#pragma unroll
        for (int i = 0; i < kTileKeys; ++i) ext = fminf(ext, s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kTileKeys; ++i) ext = i < nvis ? fminf(ext, s[i]) : ext;
      }
    }
    const float mx = nvis > 0 ? ext * sc : -INFINITY;  // the row's largest scaled score
    float alpha = 1.f;
    bool raise = false;
    if (cur.tile == 0) {
      m_ref = mx;  // every real row sees key 0; a padding row stays at -inf
    } else if (mx > m_ref + kLazyLog2) {
      raise = true;
      alpha = fast_exp2(m_ref - mx);
      m_ref = mx;
      l *= alpha;
    }
    if (__any_sync(0xffffffffu, raise)) {
      // O must hold P V of the previous tile before its rows are rescaled
      const int kp = k - 1;
      ok = mbar_wait_bounded(&sh.pv_done[kp % kPfBufs], (kp / kPfBufs) & 1, P.timeout_ns,
                             b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteSoftmaxPv, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kPfOCol + c, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_32x32b_x32(tmem + lane_base + kPfOCol + c, o);
      }
      tmem_wait_st();
    }
    // probabilities 2^(s sc - m), rounded to bf16 once: the same values feed P V and the running
    // sum; masked keys weigh 0
    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
    uint32_t pk[kTileKeys / 2];
    float ps = 0.f;
    if (all_visible) {
#pragma unroll
      for (int i = 0; i < kTileKeys / 2; ++i) {
        const uint32_t v = pack_bf16x2(fast_exp2(fmaf(s[2 * i], sc, -m_use)),
                                       fast_exp2(fmaf(s[2 * i + 1], sc, -m_use)));
        ps += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
        pk[i] = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kTileKeys / 2; ++i) {
        const float p0 = 2 * i < nvis ? fast_exp2(fmaf(s[2 * i], sc, -m_use)) : 0.f;
        const float p1 = 2 * i + 1 < nvis ? fast_exp2(fmaf(s[2 * i + 1], sc, -m_use)) : 0.f;
        const uint32_t v = pack_bf16x2(p0, p1);
        ps += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
        pk[i] = v;
      }
    }
    l += ps;
    // P over the first 32 columns of this tile's S buffer (the scores are in registers)
    tmem_st_32x32b_x32(tmem + lane_base + kPfSCol + bf * kTileKeys, pk);
    tmem_wait_st();

    const int valid = cur.L - key0;  // rows of the tile below the sequence's length
    if (valid < kTileKeys) {
      // V rows at or beyond the length may hold anything (NaN included), and 0 * NaN = NaN in
      // the MMA: zero them once the tile's copy has landed.
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

    if (cur.tile == cur.nt - 1) {
      // the unit's last tile: hand the issuer the next unit's Q (every score MMA of this unit has
      // finished: S of this tile did), then write this unit's rows once O is complete
      PfCursor nxt = cur;
      nxt.advance(P, U);
      if (!nxt.done(U)) {
        pf_write_q<D>(P, sh, nxt);
        fence_proxy_async_smem();
        mbar_arrive(sh.q_full);
      }
      ok = mbar_wait_bounded(&sh.pv_done[bf], (k / kPfBufs) & 1, P.timeout_ns, b.abort);
      if (!ok && !*b.abort) give_up(b, kSiteEpiloguePv, k);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after_sync();
      // tcgen05.ld and tcgen05.wait are warp-collective (.sync.aligned): every lane runs them,
      // padding rows included; only real rows (lim > 0) store
      const float inv = lim > 0 ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(
          P.out + ((static_cast<size_t>(cur.bi) * P.T + t_row) * P.h +
                   static_cast<size_t>(cur.j) * P.Gh + hh) * D);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kPfOCol + c, o);
        tmem_wait_ld();
        if (lim > 0) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
            dst[c / 8 + q4] = w;
          }
        }
      }
      tc_fence_before_sync();  // the O reads are done before the next unit's first P V overwrites O
    }
    cur.advance(P, U);
  }
  return true;
}

// ---------------------------------------------------------------------------------------------
// The kernel. P.G = T * Gh rows per segment (T >= 2), contiguous bf16 caches, no fused append.
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kTcThreads, kPfCtasPerSm)
    prefill_attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                const __grid_constant__ CUtensorMap tm_v, const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  TcShared sh = carve_pf_shared<D>(smem_raw);
  SharedLayout& b = sh.base;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (warp == 5) {
    tmem_alloc(sh.tmem_base, kPfTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (tid == 0) {
    *b.abort = 0;
    *b.merge = 0;
    for (int st = 0; st < pf_k_stages(D); ++st) {
      mbar_init(&b.full[st], 1);
      mbar_init(&b.empty[st], 1);
    }
    for (int st = 0; st < pf_v_stages(D); ++st) {
      mbar_init(&sh.v_full[st], 1);
      mbar_init(&sh.v_empty[st], 1);
    }
    for (int i = 0; i < kPfBufs; ++i) {
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
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sh.tmem_base;

  zero_invalid_sequences<D>(P, kTcThreads);
  const long long U = pf_units(P);

  if (warp == 4) {
    if (lane == 0) pf_produce_tiles<D>(&tm_k, &tm_v, P, sh, U);
    return;
  }
  if (warp == 5) {
    const volatile int never = 0;
    if (lane == 0) {
      const int issued = pf_issue_loop<D>(P, sh, tmem, U);
      // every MMA issued has finished, and the softmax warps are done, before the columns go
      if (issued > 0) {
        umma_commit(sh.drain);
        if (!mbar_wait_bounded(sh.drain, 0, P.drain_ns, &never)) give_up(b, kSiteDrain, 0);
      }
      if (!mbar_wait_bounded(sh.tmem_done, 0, P.drain_ns + 2 * P.timeout_ns, &never))
        give_up(b, kSiteTmemDone, 0);
    }
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kPfTmemCols);
    return;
  }
  // warps 0-3
  pf_softmax_loop<D>(P, sh, tmem, U);  // a timed-out wait has recorded itself
  tc_fence_before_sync();
  mbar_arrive(sh.tmem_done);
}

}  // namespace mqa
