// prefill_kernel.cuh -- 128-row tiles of the persistent kernel on the
// 5th-generation tensor cores (prefill and shared-prefix work; the wiki
// page's "Prefill 어텐션" section: compute-bound, chunked).
//
// Roles inside one CTA (one tile = 128 packed query rows x 128 KV tokens):
//  * warp 0 (TMA): the Q tile of an item as two 64-dim halves of a 3-D tensor
//    map over [tokens, heads, dims] -- box (64, G, 128/G) lands the G heads of
//    each token next to each other, which is the GQA row packing -- into one
//    of two Q buffers (the next item's Q loads while this one computes); per
//    KV tile one 4-D tensor-map load per page and 64-dim half of K and of V
//    ([pages, slots, heads, dims], box (64, 1, P, 1)) into a 2-stage ring,
//    128-byte swizzled; pages past the request read out of bounds and fill
//    with zeros.
//  * warp 1, one thread (MMA): S = Q K^T as 8 tcgen05.mma (M128 N128 K16,
//    both operands K-major in shared memory) into one of two S buffers in
//    tensor memory; then O += P V with P read from tensor memory (it
//    overwrites the S columns already consumed, as 16-bit pairs) and V as an
//    MN-major operand, into one of two O buffers (item parity), so an item's
//    epilogue overlaps the next item's MMAs.  S of tile j+1 is issued before
//    P V of tile j.
//  * warps 4..11 (softmax, two warpgroups): thread = query row = TMEM lane;
//    warpgroup 0 owns S/O columns 0..63, warpgroup 1 columns 64..127.  Each
//    thread loads its 64 scores once, the two halves of a row exchange their
//    maxima through shared memory (one 64-thread named barrier per lane
//    quarter), the running max moves lazily (only when it grows by more than
//    2^8, then each half rescales its O columns), P is written, and finally
//    each half reads its O columns, divides by the row sum and stores them
//    with LSE (or an fp32 partial state for a split unit).
#pragma once
#include <type_traits>

#include "attention.cuh"
#include "tc.cuh"

namespace fi {

constexpr uint32_t kQBytes = 2u * kTileM * 64u * 2u;   // two 64-dim halves of 128 rows, 16-bit
constexpr uint32_t kKVBytes = 2u * kTileN * 64u * 2u;

// Producers.  Warp 0 loads Q and K, warp 2 loads V; each walks the same tile
// stream and waits only on its own ring, so K loads run ahead of the P V work
// that frees a V stage.  The page ids of the next tile are loaded while the
// current tile's stage is awaited.
template <bool kIsV>
__device__ void pf_produce(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                           int32_t off_req) {
  const int lane = threadIdx.x & 31;
  const int G = p.group, lp = p.log2_page, P = p.page_size;
  const int ppt = kTileN >> lp;  // pages per KV tile
  const CUtensorMap* map = kIsV ? &p.tm_v : &p.tm_k;
  uint64_t* full = kIsV ? sm.v_full : sm.k_full;
  uint64_t* empty = kIsV ? sm.v_empty : sm.k_empty;
  if (lane == 0) {
    if (!kIsV) tc::prefetch_tensormap(&p.tm_q);
    tc::prefetch_tensormap(map);
  }
  uint32_t kt = 0, pe = 0;
  int q_armed[2] = {-1, -1}, armed[2] = {-1, -1};  // parity of the last armed phase
  for (int32_t i = b0; i < b1; ++i) {
    const Item it = load_item(p.iws, off_items, i);
    const Request rq = load_request(p.iws, off_req, it.b);
    const int ntiles = (it.kv1 - it.kv0 + kTileN - 1) / kTileN;
    if (ntiles == 0) continue;
    const int npages = (rq.kv_len + P - 1) >> lp;
    const int32_t* pages = p.kv_indices + rq.page_start;
    if (!kIsV) {
      const int qb = pe & 1;
      if (warp_wait(&sm.q_empty[qb], ((pe >> 1) & 1) ^ 1, &sm.abort) && lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full[qb], kQBytes);
        const int c1 = it.hk * G, c2 = rq.qo_start + it.row0 / G;
        tc::tma_load_3d(&sm.pf.q[qb][0][0][0], &p.tm_q, &sm.q_full[qb], 0, c1, c2);
        tc::tma_load_3d(&sm.pf.q[qb][1][0][0], &p.tm_q, &sm.q_full[qb], 64, c1, c2);
        q_armed[qb] = (pe >> 1) & 1;
      }
    }
    int32_t pid[4];
    auto fetch_ids = [&](int j) {
      const int pg0 = (it.kv0 + j * kTileN) >> lp;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = lane + 32 * u, pg = pg0 + e;
        pid[u] = (e < ppt && pg < npages) ? __ldg(pages + pg) : p.num_pages;  // out of bounds -> zeros
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
      if (warp_wait(&empty[st], ph ^ 1, &sm.abort)) {
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kKVBytes);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = lane + 32 * u;
          if (e < ppt) {
            uint16_t* lo = kIsV ? &sm.pf.v[st][0][e * P][0] : &sm.pf.k[st][0][e * P][0];
            uint16_t* hi = kIsV ? &sm.pf.v[st][1][e * P][0] : &sm.pf.k[st][1][e * P][0];
            tc::tma_load_4d(lo, map, &full[st], 0, it.hk, 0, cur[u]);
            tc::tma_load_4d(hi, map, &full[st], 64, it.hk, 0, cur[u]);
          }
        }
        armed[st] = ph;
      }
    }
    ++pe;
  }
  // Every load this warp armed has landed before the CTA moves on.
  if (lane == 0) {
    for (int s = 0; s < 2; ++s) {
      if (q_armed[s] >= 0) mbar_wait_drain(&sm.q_full[s], q_armed[s]);
      if (armed[s] >= 0) mbar_wait_drain(&full[s], armed[s]);
    }
  }
  __syncwarp();
}

// Single thread.  Over the CTA's stream of 128-row tiles (all its items, in
// order) it issues S = Q K^T of tile g into S buffer g % 2 and O += P V of
// tile g into its item's O buffer, whichever is ready first, polling the
// barriers without blocking; S of tile g is never issued before P V of tile
// g - 2 (it overwrites that tile's P).  An item's last S releases its Q
// buffer, its last P V publishes its O buffer.
template <typename T>
__device__ void pf_mma(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t idesc_qk = tc::idesc_f16(kBf16, false, kTileM, kTileN);
  constexpr uint32_t idesc_pv = tc::idesc_f16(kBf16, true, kTileM, kHeadDim);
  const uint32_t tmem = sm.tmem_base;
  struct Cursor {
    int32_t i;       // item index
    int ntiles, j;   // tiles of the item, tile within it
    uint32_t g, pe;  // tile in the CTA's stream, non-empty item count
  };
  auto seek = [&](Cursor& c) {  // first item with KV tiles at or after c.i
    for (; c.i < b1; ++c.i) {
      const Item it = load_item(p.iws, off_items, c.i);
      c.ntiles = (it.kv1 - it.kv0 + kTileN - 1) / kTileN;
      if (c.ntiles > 0) return;
    }
  };
  Cursor s{b0, 0, 0, 0, 0}, v{b0, 0, 0, 0, 0};
  seek(s);
  seek(v);
  bool issued = false;
  long long idle_since = clock64();
  while (v.i < b1 && !sm.abort) {
    bool progress = false;
    if (s.i < b1 && s.g <= v.g + 1) {
      const int qb = s.pe & 1, st = s.g & 1;
      if ((s.j > 0 || mbar_test_wait(&sm.q_full[qb], (s.pe >> 1) & 1)) &&
          mbar_test_wait(&sm.k_full[st], (s.g >> 1) & 1)) {
        tc::fence_after_sync();
        const uint32_t q_lo = smem_u32(&sm.pf.q[qb][0][0][0]), q_hi = smem_u32(&sm.pf.q[qb][1][0][0]);
        const uint32_t k_lo = smem_u32(&sm.pf.k[st][0][0][0]), k_hi = smem_u32(&sm.pf.k[st][1][0][0]);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 dims = 32 bytes along the swizzled 128-byte row
          const uint64_t adesc = tc::smem_desc_sw128((kk < 4 ? q_lo : q_hi) + off, 16, 1024);
          const uint64_t bdesc = tc::smem_desc_sw128((kk < 4 ? k_lo : k_hi) + off, 16, 1024);
          tc::mma_ss(tmem + st * kTileN, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.s_full[st]);
        tc::mma_commit(&sm.k_empty[st]);
        if (s.j == s.ntiles - 1) tc::mma_commit(&sm.q_empty[qb]);
        issued = progress = true;
        ++s.g;
        if (++s.j == s.ntiles) {
          s.j = 0;
          ++s.pe;
          ++s.i;
          seek(s);
        }
      }
    }
    if (v.g < s.g) {
      const int ob = v.pe & 1, st = v.g & 1;
      const uint32_t ph = (v.g >> 1) & 1;
      // the first P V of an item also needs the epilogue of the item two back to have read this O buffer
      if (mbar_test_wait(&sm.p_full[st], ph) && mbar_test_wait(&sm.v_full[st], ph) &&
          (v.j > 0 || mbar_test_wait(&sm.o_free[ob], ((v.pe >> 1) & 1) ^ 1))) {
        tc::fence_after_sync();
        const uint32_t v_lo = smem_u32(&sm.pf.v[st][0][0][0]);
        const uint32_t o_tmem = tmem + kTmemO + ob * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // V is [token][dim]: MN-major B; next 64 dims at +16 KB, next 8 tokens at +1 KB
          const uint64_t bdesc = tc::smem_desc_sw128(v_lo + kk * 16 * 128, 64 * kTileN * 2, 1024);
          // P of tokens 0..63 sits in columns 0..31 of the S buffer, tokens 64..127 in columns 64..95
          const uint32_t a_col = st * kTileN + kk * 8 + (kk >= 4 ? 32 : 0);
          tc::mma_ts(o_tmem, tmem + a_col, bdesc, idesc_pv, (v.j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.pv_done[st]);
        tc::mma_commit(&sm.v_empty[st]);
        if (v.j == v.ntiles - 1) tc::mma_commit(&sm.o_ready[ob]);
        progress = true;
        ++v.g;
        if (++v.j == v.ntiles) {
          v.j = 0;
          ++v.pe;
          ++v.i;
          seek(v);
        }
      }
    }
    if (progress) {
      idle_since = clock64();
    } else {
      __nanosleep(32);  // leave the issue slots of this SM sub-partition to the softmax warps
    }
    if (!progress && clock64() - idle_since > kWaitBudgetClocks) {
      sm.abort = kStatusTimeout;
      break;
    }
  }
  // No MMA may still run when the CTA leaves the prefill phase.
  if (issued) {
    tc::mma_commit(&sm.drain);
    mbar_wait_drain(&sm.drain, 0);
  }
}

template <typename T>
__device__ void pf_softmax(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                           int32_t off_req, int32_t off_merge, int32_t off_cnt, int causal) {
  const int sw = (threadIdx.x >> 5) - kSoftmaxWarp0;  // 0..7
  const int half = sw >> 2;                            // column half: 0 -> 0..63, 1 -> 64..127
  const int w = sw & 3;                                // == warp % 4: TMEM lanes 32w..32w+31
  const int lane = threadIdx.x & 31;
  const int r = 32 * w + lane;                         // tile row == TMEM lane
  const int tid = half * kTileM + r;                   // 0..255
  const uint32_t pair_bar = 3 + w;                     // warps 4+w and 8+w hold the same rows
  const uint32_t tl = sm.tmem_base + (uint32_t(32 * w) << 16);
  const int c0 = half * 64;
  const int G = p.group;
  const float c = p.scale_log2;
  uint32_t kt = 0, pe = 0;
  for (int32_t i = b0; i < b1; ++i) {
    const Item item = load_item(p.iws, off_items, i);
    const Request rq = load_request(p.iws, off_req, item.b);
    const int nrows = item.row1 - item.row0;
    const int ntiles = (item.kv1 - item.kv0 + kTileN - 1) / kTileN;
    const bool valid = r < nrows;
    const int row = item.row0 + r;
    const int t = row / G;
    const int head = item.hk * G + (row - t * G);
    const int64_t tok = int64_t(rq.qo_start) + t;
    int lim = -1;  // last visible KV token of this row within the chunk
    if (valid) lim = min(causal ? rq.kv_len - rq.qo_len + t : rq.kv_len - 1, item.kv1 - 1);
    float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
    bool have_o = false;
    const int ob = pe & 1;
    const uint32_t o_cols = kTmemO + ob * kHeadDim + c0;
    if (ntiles > 0) {
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t ktj = kt + j;
        const int st = ktj & 1;
        ok = ok && warp_wait(&sm.s_full[st], (ktj >> 1) & 1, &sm.abort);
        uint32_t sv[2][32];
        float mx = -INFINITY;
        const int kbase = item.kv0 + j * kTileN + c0;
        if (ok) {
          tc::fence_after_sync();
          tc::tmem_ld32(tl + st * kTileN + c0, sv[0]);
          tc::tmem_ld32(tl + st * kTileN + c0 + 32, sv[1]);
          tc::tmem_ld_wait();
          if (kbase + 63 > lim) {  // causal diagonal, chunk end or padding row: mask per element
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (kbase + h * 32 + e > lim) sv[h][e] = 0xff800000u;  // -inf
          }
          // eight independent running maxima, then a tree: no long dependency chain
          float mx8[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) mx8[a] = __uint_as_float(sv[0][a]);
#pragma unroll
          for (int e = 8; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sv[e >> 5][e & 31]));
          mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        }
        // the two halves of the row agree on its max (double-buffered by tile parity)
        sm.xmax[j & 1][half][r] = mx;
        named_barrier_sync(pair_bar, 64);
        mx = fmaxf(mx, sm.xmax[j & 1][half ^ 1][r]) * c;
        if (!ok) continue;
        const float m_new = (mx > m + kLazyRescale) ? mx : m;
        const bool rescale = (m_new != m) && have_o;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds P V of the tiles before this one: wait for the last of them
          const uint32_t prev = ktj - 1;
          ok = warp_wait(&sm.pv_done[prev & 1], (prev >> 1) & 1, &sm.abort);
          if (ok) {
            tc::fence_after_sync();
            const float alpha = rescale ? ex2(m - m_new) : 1.f;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t ov[32];
              tc::tmem_ld32(tl + o_cols + h * 32, ov);
              tc::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tc::tmem_st32(tl + o_cols + h * 32, ov);
            }
            tc::tmem_st_wait();
            if (rescale) l *= alpha;
          }
        }
        // P = 2^(s*c - m) as 16-bit pairs over the first 32 columns of this half
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;
        float sum8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) sum8[a] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a = ex2(fmaf(__uint_as_float(sv[h][2 * e]), c, -msub));
            const float b = ex2(fmaf(__uint_as_float(sv[h][2 * e + 1]), c, -msub));
            sum8[e & 7] += a + b;  // eight independent partial sums
            pk[e] = tc::pack2<T>(a, b);
          }
          tc::tmem_st16(tl + st * kTileN + c0 + h * 16, pk);
        }
        tc::tmem_st_wait();
        l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        m = m_new;
        have_o = true;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[st]);
      }
      kt += ntiles;
      ok = ok && warp_wait(&sm.o_ready[ob], (pe >> 1) & 1, &sm.abort);
      have_o = ok;
      if (ok) tc::fence_after_sync();
      ++pe;
    }
    // the row sum is the two halves' shares
    sm.xsum[i & 1][half][r] = l;  // double-buffered by item parity
    named_barrier_sync(pair_bar, 64);
    l += sm.xsum[i & 1][half ^ 1][r];
    // Epilogue, 32 columns at a time: O / l in the storage type (or the fp32
    // partial state of a split unit) and LSE in natural log.
    const bool write = valid && !sm.abort;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t ov[32];
      if (have_o) {
        tc::tmem_ld32(tl + o_cols + h * 32, ov);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      if (write) {
        const int col = c0 + h * 32;
        if (item.part < 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + col);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float* f = reinterpret_cast<const float*>(&ov[8 * e]);
            uint4 u;
            u.x = tc::pack2<T>(f[0] * inv, f[1] * inv);
            u.y = tc::pack2<T>(f[2] * inv, f[3] * inv);
            u.z = tc::pack2<T>(f[4] * inv, f[5] * inv);
            u.w = tc::pack2<T>(f[6] * inv, f[7] * inv);
            dst[e] = u;
          }
        } else {
          float4* dst =
              reinterpret_cast<float4*>(p.fws + p.partial_o_offset + (int64_t(item.part) + r) * kHeadDim + col);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                 __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
        }
      }
    }
    if (have_o) {
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_free[ob]);
    }
    if (write && half == 0) {
      if (item.part < 0) {
        if (p.lse) p.lse[tok * p.num_qo_heads + head] = lse_v;
      } else {
        p.fws[int64_t(item.part) + r] = lse_v;
      }
    }
    if (item.merge >= 0)
      merge_split_unit<T>(p, item, rq, off_merge, off_cnt, tid, kSoftmaxThreads, 2, &sm.merge_last_pf, sm.abort);
  }
}

}  // namespace fi
