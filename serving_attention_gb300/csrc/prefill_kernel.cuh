// prefill_kernel.cuh -- 128-row tiles of the persistent kernel on the
// 5th-generation tensor cores (prefill and shared-prefix work; the wiki
// page's "Prefill 어텐션" section: compute-bound, chunked).
//
// Roles inside one CTA (one tile = 128 packed query rows x 128 KV tokens):
//  * warp 0 (TMA): the Q tile once per item as two 64-dim halves of a 3-D
//    tensor map over [tokens, heads, dims] -- box (64, G, 128/G) lands the G
//    heads of each token next to each other, which is the GQA row packing --
//    then per KV tile one 4-D tensor-map load per page and 64-dim half of K
//    and of V ([pages, slots, heads, dims], box (64, 1, P, 1)), into a
//    2-stage ring, 128-byte swizzled; pages past the request read out of
//    bounds and fill with zeros.
//  * warp 1, one thread (MMA): S = Q K^T as 8 tcgen05.mma (M128 N128 K16,
//    both operands K-major in shared memory) into one of two S buffers in
//    tensor memory; then O += P V with P read from tensor memory (it
//    overwrites its S buffer as 16-bit pairs) and V as an MN-major operand.
//    S of tile j+1 is issued before P V of tile j, so the tensor core works
//    while the softmax warps work.
//  * warps 4..7 (softmax): thread = query row = TMEM lane.  Load the S row,
//    apply the bottom-right causal mask and the chunk end, move the running
//    max lazily (only when it grows by more than 2^8, then rescale O in
//    tensor memory), write P, and finally read O, divide by the row sum and
//    store O and LSE (or an fp32 partial state for a split unit).
#pragma once
#include <type_traits>

#include "attention.cuh"
#include "tc.cuh"

namespace fi {

constexpr uint32_t kQBytes = 2u * kTileM * 64u * 2u;   // two 64-dim halves of 128 rows, 16-bit
constexpr uint32_t kKVBytes = 2u * kTileN * 64u * 2u;

__device__ void pf_produce(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items,
                           int32_t off_req) {
  const int lane = threadIdx.x & 31;
  const int G = p.group, lp = p.log2_page, P = p.page_size;
  const int ppt = kTileN >> lp;  // pages per KV tile
  if (lane == 0) {
    tc::prefetch_tensormap(&p.tm_q);
    tc::prefetch_tensormap(&p.tm_k);
    tc::prefetch_tensormap(&p.tm_v);
  }
  uint32_t kt = 0, pe = 0;
  int q_armed = -1, k_armed[2] = {-1, -1}, v_armed[2] = {-1, -1};  // parity of the last armed phase
  for (int32_t i = b0; i < b1; ++i) {
    const Item it = load_item(p.iws, off_items, i);
    const Request rq = load_request(p.iws, off_req, it.b);
    const int ntiles = (it.kv1 - it.kv0 + kTileN - 1) / kTileN;
    if (ntiles == 0) continue;
    const int npages = (rq.kv_len + P - 1) >> lp;
    const int32_t* pages = p.kv_indices + rq.page_start;
    if (warp_wait(&sm.q_empty, (pe & 1) ^ 1, &sm.abort) && lane == 0) {
      mbar_arrive_expect_tx(&sm.q_full, kQBytes);
      const int c1 = it.hk * G, c2 = rq.qo_start + it.row0 / G;
      tc::tma_load_3d(&sm.pf.q[0][0][0], &p.tm_q, &sm.q_full, 0, c1, c2);
      tc::tma_load_3d(&sm.pf.q[1][0][0], &p.tm_q, &sm.q_full, 64, c1, c2);
      q_armed = pe & 1;
    }
    for (int j = 0; j < ntiles; ++j, ++kt) {
      const int st = kt & 1;
      const uint32_t ph = (kt >> 1) & 1;
      const int pg0 = (it.kv0 + j * kTileN) >> lp;
      int32_t pid[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = lane + 32 * u, pg = pg0 + e;
        pid[u] = (e < ppt && pg < npages) ? __ldg(pages + pg) : p.num_pages;  // out of bounds -> zeros
      }
      if (warp_wait(&sm.k_empty[st], ph ^ 1, &sm.abort)) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[st], kKVBytes);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = lane + 32 * u;
          if (e < ppt) {
            tc::tma_load_4d(&sm.pf.k[st][0][e * P][0], &p.tm_k, &sm.k_full[st], 0, it.hk, 0, pid[u]);
            tc::tma_load_4d(&sm.pf.k[st][1][e * P][0], &p.tm_k, &sm.k_full[st], 64, it.hk, 0, pid[u]);
          }
        }
        k_armed[st] = ph;
      }
      if (warp_wait(&sm.v_empty[st], ph ^ 1, &sm.abort)) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.v_full[st], kKVBytes);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = lane + 32 * u;
          if (e < ppt) {
            tc::tma_load_4d(&sm.pf.v[st][0][e * P][0], &p.tm_v, &sm.v_full[st], 0, it.hk, 0, pid[u]);
            tc::tma_load_4d(&sm.pf.v[st][1][e * P][0], &p.tm_v, &sm.v_full[st], 64, it.hk, 0, pid[u]);
          }
        }
        v_armed[st] = ph;
      }
    }
    ++pe;
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

// Single thread.
template <typename T>
__device__ void pf_mma(const RunParams& p, RunSmem& sm, int32_t b0, int32_t b1, int32_t off_items, int32_t off_req) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t idesc_qk = tc::idesc_f16(kBf16, false, kTileM, kTileN);
  constexpr uint32_t idesc_pv = tc::idesc_f16(kBf16, true, kTileM, kHeadDim);
  const uint32_t tmem = sm.tmem_base;
  const uint32_t q_lo = smem_u32(&sm.pf.q[0][0][0]), q_hi = smem_u32(&sm.pf.q[1][0][0]);
  uint32_t kt = 0, pe = 0;
  bool issued = false;
  for (int32_t i = b0; i < b1 && !sm.abort; ++i) {
    const Item it = load_item(p.iws, off_items, i);
    const int ntiles = (it.kv1 - it.kv0 + kTileN - 1) / kTileN;
    if (ntiles == 0) continue;
    if (!mbar_wait_bounded(&sm.q_full, pe & 1, &sm.abort)) break;
    auto issue_pv = [&](int jj) -> bool {
      const uint32_t ktj = kt + jj;
      const int st = ktj & 1;
      const uint32_t ph = (ktj >> 1) & 1;
      if (!mbar_wait_bounded(&sm.p_full[st], ph, &sm.abort)) return false;
      if (!mbar_wait_bounded(&sm.v_full[st], ph, &sm.abort)) return false;
      if (jj == 0 && !mbar_wait_bounded(&sm.o_free, (pe & 1) ^ 1, &sm.abort)) return false;
      tc::fence_after_sync();
      const uint32_t v_lo = smem_u32(&sm.pf.v[st][0][0][0]);
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk) {
        // V is [token][dim]: MN-major B; next 64 dims at +16 KB, next 8 tokens at +1 KB
        const uint64_t bdesc = tc::smem_desc_sw128(v_lo + kk * 16 * 128, 64 * kTileN * 2, 1024);
        tc::mma_ts(tmem + kTmemO, tmem + st * kTileN + kk * 8, bdesc, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
      }
      tc::mma_commit(&sm.pv_done[st]);
      tc::mma_commit(&sm.v_empty[st]);
      return true;
    };
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const uint32_t ktj = kt + j;
      const int st = ktj & 1;
      if (!mbar_wait_bounded(&sm.k_full[st], (ktj >> 1) & 1, &sm.abort)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t k_lo = smem_u32(&sm.pf.k[st][0][0][0]), k_hi = smem_u32(&sm.pf.k[st][1][0][0]);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
        const uint32_t off = (kk & 3) * 32;  // 16 dims = 32 bytes along the swizzled 128-byte row
        const uint64_t adesc = tc::smem_desc_sw128((kk < 4 ? q_lo : q_hi) + off, 16, 1024);
        const uint64_t bdesc = tc::smem_desc_sw128((kk < 4 ? k_lo : k_hi) + off, 16, 1024);
        tc::mma_ss(tmem + st * kTileN, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
      }
      issued = true;
      tc::mma_commit(&sm.s_full[st]);
      tc::mma_commit(&sm.k_empty[st]);
      if (j > 0) ok = issue_pv(j - 1);
    }
    if (ok) ok = issue_pv(ntiles - 1);
    if (!ok) break;
    tc::mma_commit(&sm.o_ready);
    tc::mma_commit(&sm.q_empty);
    kt += ntiles;
    ++pe;
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
  const int w = (threadIdx.x >> 5) - kSoftmaxWarp0;  // == warp % 4: TMEM lanes 32w..32w+31
  const int lane = threadIdx.x & 31;
  const int r = 32 * w + lane;                       // tile row == TMEM lane
  const uint32_t tl = sm.tmem_base + (uint32_t(32 * w) << 16);
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
    float m = -INFINITY, l = 0.f;
    bool have_o = false;
    if (ntiles > 0) {
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t ktj = kt + j;
        const int st = ktj & 1;
        ok = ok && warp_wait(&sm.s_full[st], (ktj >> 1) & 1, &sm.abort);
        if (!ok) continue;
        tc::fence_after_sync();
        const int kbase = item.kv0 + j * kTileN;
        const bool masked = kbase + kTileN - 1 > lim;
        // pass 1: row max over the tile, 32 columns at a time
        float mx = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t sv[32];
          tc::tmem_ld32(tl + st * kTileN + ch * 32, sv);
          tc::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = (masked && kbase + ch * 32 + e > lim) ? -INFINITY : __uint_as_float(sv[e]);
            mx = fmaxf(mx, x);
          }
        }
        mx *= c;
        const float m_new = (mx > m + kLazyRescale) ? mx : m;
        const bool rescale = (m_new != m) && (l > 0.f);
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds P V of the tiles before this one: wait for the last of them
          const uint32_t prev = ktj - 1;
          ok = warp_wait(&sm.pv_done[prev & 1], (prev >> 1) & 1, &sm.abort);
          if (ok) {
            tc::fence_after_sync();
            const float alpha = rescale ? ex2(m - m_new) : 1.f;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t ov[32];
              tc::tmem_ld32(tl + kTmemO + ch * 32, ov);
              tc::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tc::tmem_st32(tl + kTmemO + ch * 32, ov);
            }
            tc::tmem_st_wait();
            if (rescale) l *= alpha;
          }
        }
        // pass 2: P = 2^(s*c - m), 16-bit pairs written over the S columns
        // already consumed (chunk ch's P lands in columns [16ch, 16ch+16)).
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;
        float sum = 0.f;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t sv[32];
          tc::tmem_ld32(tl + st * kTileN + ch * 32, sv);
          tc::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j0 = kbase + ch * 32 + 2 * e;
            const float x0 = (masked && j0 > lim) ? -INFINITY : __uint_as_float(sv[2 * e]);
            const float x1 = (masked && j0 + 1 > lim) ? -INFINITY : __uint_as_float(sv[2 * e + 1]);
            const float a = ex2(fmaf(x0, c, -msub));
            const float b = ex2(fmaf(x1, c, -msub));
            sum += a + b;
            pk[e] = tc::pack2<T>(a, b);
          }
          tc::tmem_st16(tl + st * kTileN + ch * 16, pk);
        }
        tc::tmem_st_wait();
        l += sum;
        m = m_new;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[st]);
      }
      kt += ntiles;
      ok = ok && warp_wait(&sm.o_ready, pe & 1, &sm.abort);
      have_o = ok;
      if (ok) tc::fence_after_sync();
      ++pe;
    }
    // Epilogue, 32 columns at a time: O / l in the storage type (or the fp32
    // partial state of a split unit) and LSE in natural log.
    const bool write = valid && !sm.abort;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t ov[32];
      if (have_o) {
        tc::tmem_ld32(tl + kTmemO + ch * 32, ov);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      if (write) {
        if (item.part < 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + ch * 32);
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
          float4* dst = reinterpret_cast<float4*>(p.fws + p.partial_o_offset + (int64_t(item.part) + r) * kHeadDim +
                                                  ch * 32);
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
      if (lane == 0) mbar_arrive(&sm.o_free);
    }
    if (write) {
      if (item.part < 0) {
        if (p.lse) p.lse[tok * p.num_qo_heads + head] = lse_v;
      } else {
        p.fws[int64_t(item.part) + r] = lse_v;
      }
    }
    if (item.merge >= 0)
      merge_split_unit<T>(p, item, rq, off_merge, off_cnt, r, kTileM, 2, &sm.merge_last_pf, sm.abort);
  }
}

}  // namespace fi
