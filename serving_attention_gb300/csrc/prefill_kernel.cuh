// prefill_kernel.cuh -- prefill-class work items of the persistent kernel on
// the 5th-generation tensor cores (prefill and shared-prefix work; the wiki
// page's "Prefill 어텐션" section: compute-bound, chunked).
//
// An item is up to 256 packed query rows -- two 128-row M tiles, A and B --
// against a chunk of KV tokens walked in 128-token KV tiles.  Both M tiles use
// every K/V tile loaded, which halves the K/V bytes and the barrier round
// trips per FLOP compared with one 128-row tile per load.
//
// Roles inside one CTA:
//  * warp 0 (TMA): the item's Q tiles as 64-dim halves of a 3-D tensor map
//    over [tokens, heads, dims] -- box (64, G, 128/G) lands the G heads of
//    each token next to each other, which is the GQA row packing -- then per
//    KV tile one 4-D tensor-map load per page and 64-dim half of K
//    ([pages, slots, heads, dims], box (64, 1, P, 1)) into a 2-stage ring,
//    128-byte swizzled; pages past the request read out of bounds as zeros.
//    Warp 2 does the same for V on its own ring.
//  * warp 1 (MMA; the whole warp runs the loop, one elected lane issues):
//    S_m = Q_m K^T as 8 tcgen05.mma (M128 N128 K16, both operands K-major in
//    shared memory) into tensor memory, and
//    O_m += P_m V with P_m read back from tensor memory (it overwrites the S_m
//    columns already consumed, as 16-bit pairs) and V as an MN-major operand.
//    Order per KV tile j: P V of A for tile j, S of A for tile j+1, P V of B
//    for tile j, S of B for tile j+1 -- while one M tile's softmax runs, the
//    tensor core works on the other one.  The commit after S_m(j+1) also
//    covers P_m V(j), so a softmax that sees S_m(j+1) knows O_m is complete
//    through tile j.
//  * warps 4..7 (M tile A) and 8..11 (M tile B) (softmax): thread = query
//    row = TMEM lane, the whole 128-column S row in registers (the loaders
//    and the MMA warp give up registers for it, setmaxnreg).  Per KV tile:
//    one load of the S row, the bottom-right causal mask and the chunk end,
//    the row max; the running max moves lazily (only when it grows by more
//    than 2^8, then the O row is rescaled in tensor memory); P goes back as
//    16-bit pairs into the first 64 columns of the S buffer, in two halves
//    of 64 KV tokens with a barrier each, so P V starts on the first half
//    while the second is computed.  The two warpgroups run on different M
//    tiles, so on every SM sub-partition one warp computes while the other
//    waits.  Two row sums: one of the 16-bit P values that P V multiplies,
//    which divides O (so O weighs every key by exactly what P V used), and
//    one of the fp32 P, the exact normaliser, which gives LSE.  At the end:
//    read O, divide by its row sum, store O (a whole output tile through
//    shared memory and TMA stores) and LSE, or an fp32 partial state.
#pragma once
#include <type_traits>

#include "attention.cuh"
#include "tc.cuh"

namespace fi {

constexpr uint32_t kQTileBytes = 2u * kTileM * 64u * 2u;  // two 64-dim halves of 128 rows, 16-bit
constexpr uint32_t kKVBytes = 2u * kTileN * 64u * 2u;

__device__ __forceinline__ int item_kv_tiles(const Item& it) { return (it.kv1 - it.kv0 + kTileN - 1) / kTileN; }
__device__ __forceinline__ int item_m_tiles(const Item& it) { return it.row1 - it.row0 > kTileM ? 2 : 1; }

// Producers.  Warp 0 loads Q and K, warp 2 loads V (kProduceQK, kProduceV);
// each walks the same tile stream and waits only on its own ring.  With RoPE
// warp 0 loads all three (kProduceQKV) so that warp 2 is free to rotate.  The
// page ids of the next KV tile are loaded while the current tile's stages
// are awaited.
enum { kProduceQK = 0, kProduceV = 1, kProduceQKV = 2 };

template <int kMode>
__device__ void pf_produce(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                           int32_t off_req, int32_t num_shared) {
  constexpr bool kQK = kMode != kProduceV, kV = kMode != kProduceQK;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  if (lane == 0 && kQK) tc::prefetch_tensormap(&p.tm_q);
  if (lane < 1 + (num_shared > 0) && p.kv[lane].tc) {
    if (kQK) tc::prefetch_tensormap(&p.kv[lane].tm_k);
    if (kV) tc::prefetch_tensormap(&p.kv[lane].tm_v);
  }
  uint32_t kt = 0, pe = 0;
  int q_armed = -1, k_armed[2] = {-1, -1}, v_armed[2] = {-1, -1};  // parity of the last armed phase
  // One ring stage of K or V for the pages cur[] of the tile (one 4-D box per
  // page and 64-dim half).
  auto load_stage = [&](const CUtensorMap* map, uint64_t* full, uint16_t (*buf)[kTileN][64], int st, int hk,
                        const int32_t (&cur)[4], int P) {
    if (lane == 0) mbar_arrive_expect_tx(&full[st], kKVBytes);
    __syncwarp();
    const int ppt = kTileN / P;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = lane + 32 * u;
      if (e < ppt) {
        tc::tma_load_4d(&buf[0][e * P][0], map, &full[st], 0, hk, 0, cur[u]);
        tc::tma_load_4d(&buf[1][e * P][0], map, &full[st], 64, hk, 0, cur[u]);
      }
    }
  };
  // One item's tiles from cache kc (instantiated once per cache, so the
  // cache's fields are kernel parameters at fixed offsets).
  auto stream_item = [&](const KvCache& kc, const Item& it, int ntiles) {
    const Request& rq = it.rq;
    const int lp = kc.log2_page, P = kc.page_size;
    const int ppt = kTileN >> lp;  // pages per KV tile
    const int npages = (rq.kv_len + P - 1) >> lp;
    const int32_t* pages = kc.kv_indices + rq.page_start;
    if (kQK) {
      const int nm = item_m_tiles(it);
      if (warp_wait(&sm.q_empty, (pe & 1) ^ 1, &sm.abort) && lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, nm * kQTileBytes);
        for (int m = 0; m < nm; ++m) {
          const int c1 = it.hk * G, c2 = rq.qo_start + (it.row0 + m * kTileM) / G;
          tc::tma_load_3d(&sm.pf.q[m][0][0][0], &p.tm_q, &sm.q_full, 0, c1, c2);
          tc::tma_load_3d(&sm.pf.q[m][1][0][0], &p.tm_q, &sm.q_full, 64, c1, c2);
        }
        q_armed = pe & 1;
      }
    }
    int32_t pid[4];
    auto fetch_ids = [&](int j) {
      const int pg0 = (it.kv0 + j * kTileN) >> lp;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = lane + 32 * u, pg = pg0 + e;
        pid[u] = (e < ppt && pg < npages) ? __ldg(pages + pg) : kc.num_pages;  // out of bounds -> zeros
      }
    };
    fetch_ids(0);
    for (int j = 0; j < ntiles; ++j, ++kt) {
      const int st = kt & 1;
      const uint32_t ph = (kt >> 1) & 1;
      int32_t cur[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) cur[u] = pid[u];
      if (j + 1 < ntiles) fetch_ids(j + 1);
      if (kQK && warp_wait(&sm.k_empty[st], ph ^ 1, &sm.abort)) {
        load_stage(&kc.tm_k, sm.k_full, sm.pf.k[st], st, it.hk, cur, P);
        k_armed[st] = ph;
      }
      if (kV && warp_wait(&sm.v_empty[st], ph ^ 1, &sm.abort)) {
        load_stage(&kc.tm_v, sm.v_full, sm.pf.v[st], st, it.hk, cur, P);
        v_armed[st] = ph;
      }
    }
    ++pe;
  };
  for (int32_t i = b0; i < b1; ++i) {
    const Item it = load_item(p.iws, off_items, i);
    const int ntiles = item_kv_tiles(it);
    if (ntiles == 0) continue;
    if (it.b < num_shared)
      stream_item(p.kv[1], it, ntiles);
    else
      stream_item(p.kv[0], it, ntiles);
  }
  // Every load this warp armed has landed before the CTA moves on.
  if (lane == 0) {
    if (q_armed >= 0) mbar_wait_drain(&sm.q_full, q_armed);
    for (int s = 0; s < 2; ++s) {
      if (k_armed[s] >= 0) mbar_wait_drain(&sm.k_full[s], k_armed[s]);
      if (v_armed[s] >= 0) mbar_wait_drain(&sm.v_full[s], v_armed[s]);
    }
  }
  __syncwarp();
}

// Out of line: inlined into the kernel body, this role's code slowed the
// other tensor-core roles of the RoPE instantiation by about 9% even in
// runs where it does not execute (operands rotated by a pass).
template <typename T>
__device__ __noinline__ void pf_rope(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                                     int32_t off_req, const Variant var) {
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  // Warps 2 and 3 (the loads all go through warp 0 with RoPE).  Lane = (8-
  // frequency chunk c, position group g): positions g, g+8, g+16, ... of a
  // tile, walked two at a time with stride 8.
  constexpr int kStride = 8;
  const int c = lane & 7, g = (lane >> 3) + 4 * ((threadIdx.x >> 5) - kVWarp);
  float2 step[8];
  rope_load8(step, var.rope_table + kStride * FI_ROPE_PAIRS + 8 * c);
  __half2 amax = __float2half2_rn(0.f);
  auto rotate_row = [&](uint16_t* lo_half, uint16_t* hi_half, int row, const float2 (&cs)[8]) {
    const int pc = c ^ (row & 7);  // swizzled position of 16-byte chunk c
    uint4* plo = reinterpret_cast<uint4*>(lo_half + row * 64 + pc * 8);
    uint4* phi = reinterpret_cast<uint4*>(hi_half + row * 64 + pc * 8);
    uint4 lo = *plo, hi = *phi;
    rope_rotate8<T>(lo, hi, cs);
    absmax_f16x8(amax, lo);
    absmax_f16x8(amax, hi);
    *plo = lo;
    *phi = hi;
  };
  // Rotate `npos` consecutive positions from pos0; position u covers rows
  // [u*rpp, u*rpp + rpp) of the tile (rpp = G for Q, 1 for K), rows < nrows.
  auto rotate_tile = [&](uint16_t* lo_half, uint16_t* hi_half, int pos0, int npos, int rpp, int nrows) {
    if (g < npos) {
      float2 ca[8], cb[8];
      rope_load8(ca, var.rope_table + int64_t(pos0 + g) * FI_ROPE_PAIRS + 8 * c);
      for (int u = g; u < npos; u += 2 * kStride) {
        const bool second = u + kStride < npos;
#pragma unroll
        for (int e = 0; e < 8; ++e) cb[e] = ca[e];
        rope_advance8(cb, step);
        for (int rr = 0; rr < rpp; ++rr) {
          const int row = u * rpp + rr;
          if (row >= nrows) break;
          rotate_row(lo_half, hi_half, row, ca);
          if (second && (u + kStride) * rpp + rr < nrows) rotate_row(lo_half, hi_half, (u + kStride) * rpp + rr, cb);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) ca[e] = cb[e];
        rope_advance8(ca, step);
      }
    }
    fence_proxy_async_smem();  // the rotated operands are read by the tensor core
    __syncwarp();
  };
  uint32_t kt = 0, pe = 0;
  for (int32_t i = b0; i < b1; ++i) {
    const Item it = load_item(p.iws, off_items, i);
    const int ntiles = item_kv_tiles(it);
    if (ntiles == 0) continue;
    const Request& rq = it.rq;
    const int nrows = it.row1 - it.row0;
    const int nm = item_m_tiles(it);
    if (!warp_wait(&sm.q_full, pe & 1, &sm.abort)) break;
    for (int m = 0; m < nm; ++m) {
      // M tile m: rows m*128 .. of the item; G rows (heads) per token
      const int rows_m = min(kTileM, nrows - m * kTileM);
      const int qpos0 = rq.kv_len - rq.qo_len + (it.row0 + m * kTileM) / G;
      rotate_tile(&sm.pf.q[m][0][0][0], &sm.pf.q[m][1][0][0], qpos0, (rows_m + G - 1) / G, G, rows_m);
    }
    if (lane == 0) mbar_arrive(&sm.q_rot);
    ++pe;
    for (int j = 0; j < ntiles; ++j, ++kt) {
      const int st = kt & 1;
      if (!warp_wait(&sm.k_full[st], (kt >> 1) & 1, &sm.abort)) break;
      const int k0 = it.kv0 + j * kTileN;
      const int nk = min(kTileN, it.kv1 - k0);
      rotate_tile(&sm.pf.k[st][0][0][0], &sm.pf.k[st][1][0][0], k0, nk, 1, nk);
      if (lane == 0) mbar_arrive(&sm.k_rot[st]);
    }
  }
  if (f16x2_has_inf(amax)) atomicOr(p.iws + FI_H_STATUS, kStatusRange);
}

template <typename T, bool kRope>
__device__ void pf_mma(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  // rotated Q and K (RoPE, in the kernel or by a pass before it) are fp16
  // whatever the input type; P and V keep it
  const uint32_t idesc_qk = tc::idesc_f16(kBf16 && !kRope && !p.qk_prerotated, false, kTileM, kTileN);
  constexpr uint32_t idesc_pv = tc::idesc_f16(kBf16, true, kTileM, kHeadDim);
  const int lane = threadIdx.x & 31;
  const uint32_t tmem = sm.tmem_base;
  // Shared-memory descriptors of the first block of each operand buffer; the
  // start-address field counts 16-byte units, so the other blocks and the K16
  // steps are constant offsets: a 64-dim half is 16 KB (1024 units), an M
  // tile or ring stage 32 KB (2048), 16 dims along a swizzled row 32 bytes
  // (2), 16 V tokens 2 KB (128).  Every sum is a real shared-memory address,
  // which stays below 2^18 bytes: the field never carries.
  const uint64_t dq = tc::smem_desc_sw128(smem_u32(&sm.pf.q[0][0][0][0]), 16, 1024);
  const uint64_t dk = tc::smem_desc_sw128(smem_u32(&sm.pf.k[0][0][0][0]), 16, 1024);
  const uint64_t dv = tc::smem_desc_sw128(smem_u32(&sm.pf.v[0][0][0][0]), 64 * kTileN * 2, 1024);
  uint32_t kt = 0, pe = 0;       // KV tiles and non-empty items so far
  uint32_t tiles_m[2] = {0, 0};  // per M tile: P V issued so far (phases of p_full)
  uint32_t items_m[2] = {0, 0};  // per M tile: items finished (phases of o_free)
  bool issued = false;
  auto issue_s = [&](int m, int st) {
    const uint64_t a0 = dq + 2048u * m, b0k = dk + 2048u * st;
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t step = 1024u * (kk >> 2) + 2u * (kk & 3);
      tc::mma_ss_warp(tmem + m * kTileN, a0 + step, b0k + step, idesc_qk, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit_warp(&sm.s_full[m]);
    issued = true;
  };
  auto issue_pv = [&](int m, int st, bool first, int half) {
    // V is [token][dim]: MN-major B; next 64 dims at +16 KB, next 8 tokens at +1 KB
    const uint64_t bv = dv + 2048u * st;
    const uint32_t o_tmem = tmem + kTmemO + m * kHeadDim;
#pragma unroll
    for (int kk = 4 * half; kk < 4 * half + 4; ++kk) {
      // P_m of tokens 16kk..16kk+15: columns 8kk..8kk+7 of the S_m buffer, 16-bit pairs
      tc::mma_ts_warp(o_tmem, tmem + m * kTileN + kk * 8, bv + 128u * kk, idesc_pv, (!first || kk > 0) ? 1u : 0u);
    }
  };
  for (int32_t i = b0; i < b1; ++i) {
    if (__shfl_sync(0xffffffffu, sm.abort, 0)) break;
    const Item it = load_item(p.iws, off_items, i);
    const int ntiles = item_kv_tiles(it);
    if (ntiles == 0) continue;
    const int nm = item_m_tiles(it);
    // with RoPE the operands are read once the rotation warp has released them
    // (operands rotated by a pass before the run arrive ready: the plain waits)
    const bool rot_roles = kRope && !p.qk_prerotated;
    uint64_t* const q_bar = rot_roles ? &sm.q_rot : &sm.q_full;
    uint64_t* const k_bars = rot_roles ? sm.k_rot : sm.k_full;
    bool ok = warp_wait_all(2, q_bar, pe & 1, &k_bars[kt & 1], (kt >> 1) & 1, nullptr, 0, nullptr, 0, &sm.abort);
    if (!ok) break;
    tc::fence_after_sync();
    for (int m = 0; m < nm; ++m) issue_s(m, kt & 1);
    tc::mma_commit_warp(&sm.k_empty[kt & 1]);
    if (ntiles == 1) tc::mma_commit_warp(&sm.q_empty);  // the item's last read of Q
    for (int j = 0; j < ntiles && ok; ++j) {
      const uint32_t g = kt + j;  // KV tile in the CTA's stream
      const int st = g & 1;
      const bool more = j + 1 < ntiles;
      const int st_next = (g + 1) & 1;
      for (int m = 0; m < nm && ok; ++m) {
        // Everything this step reads, polled at once: P_m of tile j (tokens
        // 0..63); for M tile A also V of tile j and K of tile j+1; at an
        // item's first tile the O_m columns.  Entries that do not apply
        // repeat the first.  The second half of P is awaited on its own, so
        // the first four P V steps overlap the end of the softmax.
        uint64_t* const pb = &sm.p_full[m][0];
        const uint32_t pp = tiles_m[m] & 1;
        const bool kv = m == 0, need_k = kv && more;
        ok = warp_wait_all(4, pb, pp, kv ? &sm.v_full[st] : pb, kv ? (g >> 1) & 1 : pp,
                           j == 0 ? &sm.o_free[m] : pb, j == 0 ? (items_m[m] & 1) ^ 1 : pp,
                           need_k ? &k_bars[st_next] : pb, need_k ? ((g + 1) >> 1) & 1 : pp, &sm.abort);
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv(m, st, j == 0, 0);
        ok = warp_wait(&sm.p_full[m][1], pp, &sm.abort);
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv(m, st, false, 1);
        ++tiles_m[m];
        if (!more) {
          tc::mma_commit_warp(&sm.o_ready[m]);
          continue;
        }
        issue_s(m, st_next);
      }
      if (!ok) break;
      tc::mma_commit_warp(&sm.v_empty[st]);
      if (more) {
        tc::mma_commit_warp(&sm.k_empty[st_next]);
        if (j + 2 == ntiles) tc::mma_commit_warp(&sm.q_empty);
      }
    }
    if (!ok) break;
    for (int m = 0; m < nm; ++m) ++items_m[m];
    kt += ntiles;
    ++pe;
  }
  // No MMA may still run when the CTA leaves the prefill phase.
  if (issued) {
    tc::mma_commit_warp(&sm.drain);
    if (lane == 0) mbar_wait_drain(&sm.drain, 0);
    __syncwarp();
  }
}

template <typename T, bool kCap, bool kMask>
__device__ void pf_softmax(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                           int32_t off_req, int32_t off_merge, int32_t off_cnt, int causal, int32_t num_shared,
                           const Variant var) {
  const int sw = (threadIdx.x >> 5) - kSoftmaxWarp0;  // 0..7
  const int mt = sw >> 2;                              // this warpgroup's M tile: 0 = A, 1 = B
  const int w = sw & 3;                                // == warp % 4: TMEM lanes 32w..32w+31
  const int lane = threadIdx.x & 31;
  const int r = 32 * w + lane;                         // row within the M tile == TMEM lane
  const int tid = mt * kTileM + r;                     // 0..255
  const uint32_t tl = sm.tmem_base + (uint32_t(32 * w) << 16);
  const uint32_t s_cols = tl + mt * kTileN, o_cols = tl + kTmemO + mt * kHeadDim;
  const int G = p.group;
  const float c = p.scale_log2;
  const float cs = kCap ? var.cap_a : c;  // log2-domain factor of the (tanh of the) logits
  uint32_t tiles = 0, items = 0;  // phases of s_full[mt] and o_ready[mt]
  for (int32_t i = b0; i < b1; ++i) {
    const Item item = load_item(p.iws, off_items, i);
    const Request& rq = item.rq;
    const int nrows = item.row1 - item.row0;
    const int ntiles = item_kv_tiles(item);
    const int prow = mt * kTileM + r;  // packed row within the item
    if (mt < item_m_tiles(item)) {
      int lim = -1, lo = 0;  // visible KV tokens of this row: [lo, lim] and the sink (lim -1: padding row)
      if (prow < nrows) {
        const int t = (item.row0 + prow) / G;
        const bool causal_i = causal && item.b >= num_shared;  // a shared block's keys are all visible
        lim = min(causal_i ? rq.kv_len - rq.qo_len + t : rq.kv_len - 1, item.kv1 - 1);
        if (kMask) lo = window_low(var, rq.kv_len - rq.qo_len + t);
      }
      // lrun: sum of the fp32 P (the exact normaliser, for LSE); lrun_r: sum
      // of the 16-bit P that P V multiplies (the normaliser of O)
      float mrun = -INFINITY, lrun = 0.f, lrun_r = 0.f;
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        ok = ok && warp_wait(&sm.s_full[mt], tiles & 1, &sm.abort);
        ++tiles;
        if (!ok) continue;
        tc::fence_after_sync();
        uint32_t sv[4][32];
#pragma unroll
        for (int h = 0; h < 4; ++h) tc::tmem_ld32(s_cols + 32 * h, sv[h]);
        tc::tmem_ld_wait();
        const int kbase = item.kv0 + j * kTileN;
        if (kCap) {  // tanh(scale * s / cap), which cs = cap * log2(e) turns into the capped log2-domain logit
          const float kb = c * var.cap_b * 0.34657359f;  // scale * log2(e) * (2 / cap) * ln(2) / 2 = scale / cap
          const float2 kb2 = make_float2(kb, kb), zero = make_float2(0.f, 0.f);
#pragma unroll
          for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y = fma2(make_float2(__uint_as_float(sv[h][e]), __uint_as_float(sv[h][e + 1])), kb2, zero);
              sv[h][e] = __float_as_uint(tanh_approx(y.x));
              sv[h][e + 1] = __float_as_uint(tanh_approx(y.y));
            }
        }
        if (kbase + kTileN - 1 > lim || (kMask && kbase < lo)) {  // causal diagonal, chunk end, padding row, window
#pragma unroll
          for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int key = kbase + 32 * h + e;
              if (key > lim || (kMask && key < lo && key >= var.sink)) sv[h][e] = 0xff800000u;  // -inf
            }
        }
        // row max in eight independent chains of three-input maxima
        auto sval = [&](int e) { return __uint_as_float(sv[e >> 5][e & 31]); };
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = sval(a);
#pragma unroll
        for (int e = 8; e + 16 <= kTileN; e += 16)
#pragma unroll
          for (int a = 0; a < 8; ++a) mx8[a] = max3(mx8[a], sval(e + a), sval(e + 8 + a));
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(mx8[a], sval(kTileN - 8 + a));
        const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * cs;
        const float m_old = mrun;
        const float m_new = (mx > m_old + kLazyRescale) ? mx : m_old;
        const bool rescale = (m_new != m_old) && j > 0;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds P V of every earlier tile (covered by this S's commit)
          const float alpha = rescale ? ex2(m_old - m_new) : 1.f;
#pragma unroll 1
          for (int h = 0; h < 4; ++h) {
            uint32_t ov[32];
            tc::tmem_ld32(o_cols + 32 * h, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tc::tmem_st32(o_cols + 32 * h, ov);
          }
          tc::tmem_st_wait();
          if (rescale) {
            lrun *= alpha;
            lrun_r *= alpha;
          }
        }
        // P = 2^(s*c - m) as 16-bit pairs over the first 64 columns of the S
        // buffer, published in two halves of 64 KV tokens each
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;
        const float2 cc = make_float2(cs, cs), nms = make_float2(-msub, -msub);
        float2 sum4[4], sumr[2];
#pragma unroll
        for (int a = 0; a < 4; ++a) sum4[a] = make_float2(0.f, 0.f);
        sumr[0] = sumr[1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int h = 2 * half; h < 2 * half + 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x =
                  fma2(make_float2(__uint_as_float(sv[h][2 * e]), __uint_as_float(sv[h][2 * e + 1])), cc, nms);
              const float2 pe = make_float2(ex2(x.x), ex2(x.y));
              sum4[e & 3] = add2(sum4[e & 3], pe);
              pk[e] = tc::pack2<T>(pe.x, pe.y);
              tc::add_packed2<T>(sumr[e & 1], pk[e]);
            }
            tc::tmem_st16(s_cols + 16 * h, pk);
          }
          tc::tmem_st_wait();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.p_full[mt][half]);
        }
        const float2 s01 = add2(sum4[0], sum4[1]), s23 = add2(sum4[2], sum4[3]), s4 = add2(s01, s23);
        lrun += s4.x + s4.y;
        const float2 sr = add2(sumr[0], sumr[1]);
        lrun_r += sr.x + sr.y;
        mrun = m_new;
      }
      // Epilogue: O / l in the storage type (or the fp32 partial state of a
      // split unit), LSE in natural log.  The O row leaves tensor memory in
      // one load, and the O columns go back to the MMA warp right away.
      bool have_o = false;
      if (ntiles > 0) {
        ok = ok && warp_wait(&sm.o_ready[mt], items & 1, &sm.abort);
        ++items;
        have_o = ok;
      }
      uint32_t ov[4][32];
      if (have_o) {
        tc::fence_after_sync();
#pragma unroll
        for (int h = 0; h < 4; ++h) tc::tmem_ld32(o_cols + 32 * h, ov[h]);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_free[mt]);
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[h][e] = 0u;
      }
      const bool write = prow < nrows && !sm.abort;
      const int row = item.row0 + prow;
      const int t = row / G;
      const int head = item.hk * G + (row - t * G);
      const int64_t tok = int64_t(rq.qo_start) + t;
      const float inv = lrun_r > 0.f ? 1.f / lrun_r : 0.f;
      const float lse_v = lrun > 0.f ? (mrun + __log2f(lrun)) * 0.69314718055994531f : -INFINITY;
      auto pack8 = [&](int h, int e0) {  // 8 normalised values as 16-bit pairs
        uint4 u;
        u.x = tc::pack2<T>(__uint_as_float(ov[h][e0]) * inv, __uint_as_float(ov[h][e0 + 1]) * inv);
        u.y = tc::pack2<T>(__uint_as_float(ov[h][e0 + 2]) * inv, __uint_as_float(ov[h][e0 + 3]) * inv);
        u.z = tc::pack2<T>(__uint_as_float(ov[h][e0 + 4]) * inv, __uint_as_float(ov[h][e0 + 5]) * inv);
        u.w = tc::pack2<T>(__uint_as_float(ov[h][e0 + 6]) * inv, __uint_as_float(ov[h][e0 + 7]) * inv);
        return u;
      };
      if (item.part < 0 && (mt + 1) * kTileM <= nrows) {
        // A whole 128-row tile of an unsplit item leaves through shared
        // memory: per d half, each thread writes its row as 128 bytes in the
        // 128-byte swizzled layout of the Q tile, then one thread of the
        // warpgroup stores the box (64 dims, G heads, 128/G tokens) with TMA.
        const uint32_t wg_bar = kEpilogueBarrier0 + mt;
        uint16_t* stage = &sm.pf.ostage[mt][0][0];
        uint4* my_row = reinterpret_cast<uint4*>(stage + r * 64);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int cch = 0; cch < 8; ++cch) my_row[cch ^ (r & 7)] = pack8(2 * half + (cch >> 2), 8 * (cch & 3));
          fence_proxy_async_smem();
          named_barrier_sync(wg_bar, 128);
          if ((threadIdx.x & 127) == 0 && !sm.abort) {
            tc::tma_store_3d(&p.tm_o, stage, 64 * half, item.hk * G, rq.qo_start + (item.row0 + mt * kTileM) / G);
            tc::bulk_commit();
            tc::bulk_wait_read_all();  // the staging rows may be written again
          }
          named_barrier_sync(wg_bar, 128);
        }
      } else if (write) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int col = 32 * h;
          if (item.part < 0) {
            uint4* dst =
                reinterpret_cast<uint4*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + col);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = pack8(h, 8 * e);
          } else {
            float4* dst = reinterpret_cast<float4*>(p.fws + p.partial_o_offset +
                                                    (int64_t(item.part) + prow) * kHeadDim + col);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(ov[h][4 * e]) * inv, __uint_as_float(ov[h][4 * e + 1]) * inv,
                                   __uint_as_float(ov[h][4 * e + 2]) * inv, __uint_as_float(ov[h][4 * e + 3]) * inv);
          }
        }
      }
      if (write) {
        if (item.part < 0) {
          if (p.lse) p.lse[tok * p.num_qo_heads + head] = lse_v;
        } else {
          p.fws[int64_t(item.part) + prow] = lse_v;
        }
      }
    }
    if (item.merge >= 0)
      merge_split_unit<T>(p, item, rq, off_merge, off_cnt, tid, kSoftmaxThreads, 2, &sm.merge_last_pf, sm.abort);
  }
  if ((threadIdx.x & 127) == 0) tc::bulk_wait_all();  // output tiles written before the CTA moves on
}

}  // namespace fi
