// attention_kernel.cuh -- persistent paged-attention kernel, CUDA-core path.
//
// One CTA per SM walks its slice of the planned work list (the plan/run split
// of the FlashInfer paper summary, "3. 동적 부하 분산 스케줄링").  Per item
// (request b, KV head hk, packed query rows [row0,row1), KV tokens [kv0,kv1)):
//
//  * warp 0 streams the chunk's K and V, 128 tokens per stage, into a 3-deep
//    shared-memory ring: one TMA box per page and tensor, completion counted
//    in bytes on the stage's mbarrier (see produce()).  Each K/V row of one
//    head is 256 contiguous bytes.  A multi-head item (one query token, pages
//    of one token) takes H KV heads at once: a stage then holds 128 / H
//    tokens, each token's H rows brought by one box.
//  * warps 4..11 hold the G query heads that share KV head hk (GQA packing,
//    wiki page "Decode 어텐션") in registers, 4 packed rows per half-warp,
//    and score every KV token read from shared memory once for all of them.
//    A half-warp owns one token at a time (16 lanes x 8 dims); partial dot
//    products are reduced with a 5-shuffle butterfly that leaves each lane
//    the full score of one row.  Softmax is online with a lazily moved
//    running max (log2 domain).
//  * a multi-head item's 32 packed rows are the G query heads of each of its
//    H KV heads; each row group of 4 lies in one KV head and scores that
//    head's rows of the stage.
//  * the half-warps' states are merged in shared memory; an unsplit item
//    writes O (storage type) and LSE (natural log), a split item writes its
//    fp32 partial state, and the CTA that finishes the last chunk of a split
//    unit merges the unit's partials in chunk order (no inter-CTA waits).
#pragma once
#include <type_traits>

#include "attention.cuh"
#include "tc.cuh"

namespace fi {

__device__ __forceinline__ int32_t ws_header(const int32_t* iws, int f) { return __ldg(iws + f); }

// Row group layout of one pass: ng groups of 4 rows (ng a power of two),
// 8/ng consumer warps share a group and split its tokens.
__device__ __forceinline__ int groups_in_pass(int rows) {
  int g = (rows + kRowsPerGroup - 1) / kRowsPerGroup;
  return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
}

// ---------------------------------------------------------------- producer

// K and V of one stage: 128 tokens of one KV head.  One unswizzled 4-D TMA box
// (128 dims, 1 head, min(P, 128) slots, 1 page) per page and tensor, issued by
// lane (box % 32); a multi-head item's stage is 128 / H tokens of H heads,
// one box (128 dims, H heads, 1 slot, 1 page) per token and tensor, rows
// token-major.  The page ids of the next stage are loaded one stage ahead
// into the issuing lanes' registers (the wiki page's page-index prefetch,
// "1) 블록-스파스 KV 포맷").  Pages past the chunk (which need not fill its last
// stage) are addressed out of bounds and arrive as zeros without a read of
// HBM; stage tokens past the chunk are masked
// by the consumers.
static __device__ void produce(const RunParams& p, RunSmem& sm, int32_t item_begin, int32_t item_end, int32_t off_items,
                        int32_t off_req, int32_t num_shared) {
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kStageBytes = 2u * kStageTokens * kHeadDim * 2u;
  if (lane < 1 + (num_shared > 0)) {
    const KvCache& kc = p.kv[lane];
    tc::prefetch_tensormap(kc.gather_rows ? &kc.tm_kg : &kc.tm_kd);
    tc::prefetch_tensormap(kc.gather_rows ? &kc.tm_vg : &kc.tm_vd);
  } else if (lane == 2 && p.kv[0].mh_heads) {
    tc::prefetch_tensormap(&p.kv[0].tm_kh);
    tc::prefetch_tensormap(&p.kv[0].tm_vh);
  }
  uint32_t it = 0;
  int armed[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) armed[s] = -1;
  const int G = p.group;
  // Near the end of an item (its last stage issued, the consumers at most a
  // ring behind), the next item's query rows and first page ids are brought
  // into L2, so that neither the consumers' query load nor this warp's page-id
  // load at the next item start waits on HBM.
  auto prefetch_next = [&](const Item& nx) {
    const int lines = (nx.row1 - nx.row0) * 2;  // two 128-byte lines per packed row
    for (int l = lane; l < lines; l += 32) {
      const int row = nx.row0 + (l >> 1);
      const int t = row_token(nx, row, G);
      tc::prefetch_l2(p.q + (int64_t(nx.rq.qo_start) + t) * p.q_stride_tok +
                      int64_t(nx.hk * G + row - t * G) * p.q_stride_head + (l & 1) * 64);
    }
    if (lane == 0) {
      const KvCache& kn = cache_of(p, nx.b, num_shared);
      tc::prefetch_l2(kn.kv_indices + nx.rq.page_start + (nx.kv0 >> kn.log2_page));
    }
  };
  // One item's stages from cache kc (instantiated once per cache, so the
  // cache's fields are kernel parameters at fixed offsets).
  auto stream_item = [&](const KvCache& kc, const Item& item, const Item* nx) {
    const Request& rq = item.rq;
    const int lp = kc.log2_page, P = kc.page_size;
    const int H = item.heads;             // a multi-head item (page size 1): H KV heads per token
    const int stok = kStageTokens / H;    // tokens per stage
    const bool gather = kc.gather_rows && H == 1;
    const int boxes = H > 1 ? stok : P >= kStageTokens ? 1 : (kStageTokens >> lp);  // per stage and tensor
    const int box_slots = P >= kStageTokens ? kStageTokens : P;
    const int nrows = item.row1 - item.row0;
    const int passes = (nrows + kRowsPerPass - 1) / kRowsPerPass;
    const int nst = (item.kv1 - item.kv0 + stok - 1) / stok;
    const int npages = min((rq.kv_len + P - 1) >> lp, (item.kv1 + P - 1) >> lp);  // pages the chunk touches
    const int32_t* pages = kc.kv_indices + rq.page_start;
    for (int pass = 0; pass < passes; ++pass) {
      // page ids of the next stage's boxes: lane, lane + 32, ... (box loads)
      // or 4 * lane .. 4 * lane + 3 (the four rows of a lane's gather)
      int32_t nxid[kBoxLanes];
      auto fetch_ids = [&](int st) {
        const int pg0 = (item.kv0 + st * stok) >> lp;
#pragma unroll
        for (int r = 0; r < kBoxLanes; ++r) {
          const int bx = gather ? kBoxLanes * lane + r : lane + 32 * r;
          nxid[r] = (bx < boxes && pg0 + bx < npages) ? __ldg(pages + pg0 + bx) : kc.num_pages;
        }
      };
      if (nst > 0) fetch_ids(0);
      for (int st = 0; st < nst; ++st, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        int32_t id[kBoxLanes];
#pragma unroll
        for (int r = 0; r < kBoxLanes; ++r) id[r] = nxid[r];
        if (st + 1 < nst) fetch_ids(st + 1);
        if (!warp_wait(&sm.empty[s], ph ^ 1, &sm.abort)) continue;
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
        __syncwarp();
        const int j0 = item.kv0 + st * stok;
        const int slot0 = P > kStageTokens ? (j0 & (P - 1)) : 0;
        if (H > 1) {
          // multi-head item: one box per token and tensor with the token's
          // rows of KV heads hk .. hk + H - 1 (H * 256 contiguous bytes of
          // the stage, token-major: stage row = token * H + head offset)
#pragma unroll
          for (int r = 0; r < kBoxLanes; ++r) {
            const int bx = lane + 32 * r;
            if (bx < boxes) {
              tc::tma_load_4d(&sm.dec.k[s][bx * H][0], &kc.tm_kh, &sm.full[s], 0, item.hk, 0, id[r]);
              tc::tma_load_4d(&sm.dec.v[s][bx * H][0], &kc.tm_vh, &sm.full[s], 0, item.hk, 0, id[r]);
            }
          }
        } else if (gather) {
          // page size 1: lane l brings tokens 4l..4l+3 of K and of V with one
          // four-row gather each (row page * rows_per_page + hk; pages past
          // the chunk are rows past the tensor and arrive as zeros)
          static_assert(kBoxLanes == 4, "one four-row gather per lane and tensor");
          const int rk = kc.gather_rows_k, rv = kc.gather_rows_v;
          tc::tma_gather4_2d(&sm.dec.k[s][4 * lane][0], &kc.tm_kg, &sm.full[s], 0, id[0] * rk + item.hk,
                             id[1] * rk + item.hk, id[2] * rk + item.hk, id[3] * rk + item.hk);
          tc::tma_gather4_2d(&sm.dec.v[s][4 * lane][0], &kc.tm_vg, &sm.full[s], 0, id[0] * rv + item.hk,
                             id[1] * rv + item.hk, id[2] * rv + item.hk, id[3] * rv + item.hk);
        } else {
#pragma unroll
          for (int r = 0; r < kBoxLanes; ++r) {
            const int bx = lane + 32 * r;
            if (bx < boxes) {
              tc::tma_load_4d(&sm.dec.k[s][bx * box_slots][0], &kc.tm_kd, &sm.full[s], 0, item.hk, slot0, id[r]);
              tc::tma_load_4d(&sm.dec.v[s][bx * box_slots][0], &kc.tm_vd, &sm.full[s], 0, item.hk, slot0, id[r]);
            }
          }
        }
        armed[s] = ph;
        if (nx && st + 1 == nst && pass + 1 == passes) prefetch_next(*nx);
      }
    }
  };
  Item next = item_begin < item_end ? load_item(p.iws, off_items, item_begin) : Item{};
  for (int32_t i = item_begin; i < item_end; ++i) {
    const Item item = next;
    const bool more = i + 1 < item_end;
    if (more) next = load_item(p.iws, off_items, i + 1);
    if (item.b < num_shared)
      stream_item(p.kv[1], item, more ? &next : nullptr);
    else
      stream_item(p.kv[0], item, more ? &next : nullptr);
  }
  // Every load this warp armed has landed before the CTA moves on.
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s)
      if (armed[s] >= 0) mbar_wait_drain(&sm.full[s], armed[s]);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- split merge

// Split unit: every chunk wrote its fp32 partial state; the CTA whose
// atomic increment completes the unit's counter merges the chunks in chunk
// order (deterministic), writes O and LSE, and resets the counter.  No CTA
// ever waits for another.  `nthreads` threads with index `tid` take part and
// synchronise on named barrier `bar`; the barrier sequence depends only on
// the plan, never on the abort flag, so all participating warps pass it.
// Units the plan marks late (prefill-class tiles, up to 256 rows) are left to
// the row-parallel merge launched after the run, when one follows: one SM
// reading all their partial states would hold the run's end back.
template <typename T>
__device__ void merge_split_unit(const RunParams& p, const Item& item, const Request& rq, int32_t off_merge,
                                 int32_t off_cnt, int tid, int nthreads, int bar, int* flag, int aborted) {
  if (p.late_merge && __ldg(p.iws + off_merge + FI_MERGE_INTS * item.merge + FI_MERGE_LATE)) return;
  const int G = p.group;
  const int nrows = item.row1 - item.row0;
  __threadfence();
  named_barrier_sync(bar, nthreads);
  if (tid == 0) {
    int last = 0;
    if (!aborted) {
      const int32_t n = __ldg(p.iws + off_merge + FI_MERGE_INTS * item.merge + 4);
      const int old = atomicAdd(p.iws + off_cnt + item.merge, 1);
      last = (old == n - 1);
    }
    *reinterpret_cast<volatile int*>(flag) = last;
  }
  named_barrier_sync(bar, nthreads);
  if (*reinterpret_cast<volatile int*>(flag)) {
    __threadfence();
    const int32_t* mu = p.iws + off_merge + FI_MERGE_INTS * item.merge;
    const int n = __ldg(mu + 4);
    const int base = __ldg(mu + 5);
    for (int task = tid; task < nrows * 32; task += nthreads) {
      const int pr = task >> 5, ch = task & 31;
      float M = -INFINITY;
      for (int c = 0; c < n; ++c) M = fmaxf(M, __ldcg(p.fws + base + c * nrows + pr));
      float Ls = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
        for (int c = 0; c < n; ++c) {
          const int64_t prw = int64_t(base) + c * nrows + pr;
          const float w = ex2((__ldcg(p.fws + prw) - M) * 1.4426950408889634f);
          const float4 v = __ldcg(reinterpret_cast<const float4*>(p.fws + p.partial_o_offset + prw * kHeadDim) + ch);
          Ls += w;
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const int row = item.row0 + pr;
      const int t = row_token(item, row, G);
      const int head = item.hk * G + (row - t * G);
      const int64_t tok = rq.qo_start + t;
      uint2 packed;
      packed.x = Elem<T>::from_float2(acc.x * inv, acc.y * inv);
      packed.y = Elem<T>::from_float2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + ch * 4) = packed;
      if (ch == 0 && p.lse) p.lse[tok * p.num_qo_heads + head] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
    }
    if (tid == 0) p.iws[off_cnt + item.merge] = 0;  // ready for the next run of this plan
  }
  named_barrier_sync(bar, nthreads);
}

// ---------------------------------------------------------------- consumer

// Sum of v[0..3] over the 16 lanes of a half-warp, leaving lane L with the
// sum of row (L >> 2) & 3: two exchange steps that halve the number of values
// each lane carries, then two plain butterfly steps.
__device__ __forceinline__ float reduce_rows4(float v0, float v1, float v2, float v3, int lane16) {
  const bool hi8 = lane16 & 8;
  float a0 = hi8 ? v2 : v0, a1 = hi8 ? v3 : v1;
  const float b0 = hi8 ? v0 : v2, b1 = hi8 ? v1 : v3;
  a0 += __shfl_xor_sync(0xffffffffu, b0, 8);
  a1 += __shfl_xor_sync(0xffffffffu, b1, 8);
  const bool hi4 = lane16 & 4;
  float keep = hi4 ? a1 : a0;
  const float send = hi4 ? a0 : a1;
  keep += __shfl_xor_sync(0xffffffffu, send, 4);
  keep += __shfl_xor_sync(0xffffffffu, keep, 2);
  keep += __shfl_xor_sync(0xffffffffu, keep, 1);
  return keep;
}

// 8 storage elements -> 4 fp32 pairs (element 2i in .x, 2i+1 in .y).
template <typename T>
__device__ __forceinline__ void unpack4x2(const uint4& u, float2 (&f)[4]) {
  f[0] = Elem<T>::to_float2(u.x);
  f[1] = Elem<T>::to_float2(u.y);
  f[2] = Elem<T>::to_float2(u.z);
  f[3] = Elem<T>::to_float2(u.w);
}

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const float2 a = Elem<T>::to_float2(u.x), b = Elem<T>::to_float2(u.y);
  const float2 c = Elem<T>::to_float2(u.z), d = Elem<T>::to_float2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  u.x = Elem<T>::from_float2(f[0], f[1]);
  u.y = Elem<T>::from_float2(f[2], f[3]);
  u.z = Elem<T>::from_float2(f[4], f[5]);
  u.w = Elem<T>::from_float2(f[6], f[7]);
  return u;
}

// RoPE of 8 dim pairs in 16-bit storage: lo holds dims i..i+7 of the first
// half of a head, hi dims i+64..i+71; cs the (cos, sin) of their 8 angles.
// x_i' = x_i cos - x_{i+64} sin, x_{i+64}' = x_{i+64} cos + x_i sin, in fp32,
// rounded once to fp16 whatever the input type: fp16 keeps 11 significant
// bits where bf16 keeps 8, and the rotated q and k meet only each other
// (S = q.k), so the score does not carry a bf16 rounding of the rotation.
// Rotated values must stay inside the fp16 range (|x| <= 65504): every role
// and pass that rotates into fp16 keeps a running maximum (absmax_f16x8)
// and records kStatusRange when it reaches inf.  (TOut other than fp16: the
// standalone rotation utilities, which write the input's own type.)
template <typename T, typename TOut = __half>
__device__ __forceinline__ void rope_rotate8(uint4& lo, uint4& hi, const float2 (&cs)[8]) {
  float a[8], b[8];
  unpack8<T>(lo, a);
  unpack8<T>(hi, b);
  float ra[8], rb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ra[e] = fmaf(a[e], cs[e].x, -b[e] * cs[e].y);
    rb[e] = fmaf(b[e], cs[e].x, a[e] * cs[e].y);
  }
  lo = pack8<TOut>(ra);
  hi = pack8<TOut>(rb);
}

// Range guard of the fp16 rotation: m = max(m, |x|) over the eight fp16
// values of u (packed max; an input NaN is passed over, an overflow to inf
// is kept), and whether a running maximum has reached inf.
__device__ __forceinline__ void absmax_f16x8(__half2& m, const uint4& u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __half2 h;
    memcpy(&h, &w[k], 4);
    m = __hmax2(m, __habs2(h));
  }
}

__device__ __forceinline__ bool f16x2_has_inf(__half2 m) {
  return __hisinf(__low2half(m)) != 0 || __hisinf(__high2half(m)) != 0;
}

// (cos, sin) of 8 consecutive frequencies of one position: 64 bytes of the table.
__device__ __forceinline__ void rope_load8(float2 (&cs)[8], const float2* __restrict__ p) {
  const float4* p4 = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 t = __ldg(p4 + k);
    cs[2 * k] = make_float2(t.x, t.y);
    cs[2 * k + 1] = make_float2(t.z, t.w);
  }
}

// Angles of the next position of a walk with a fixed stride: multiply by the
// stride's (cos, sin) (angle addition), so a walk needs only its first row
// and the stride's row from the table; fp32 drift over 32 steps is ~1e-6.
__device__ __forceinline__ void rope_advance8(float2 (&cs)[8], const float2 (&step)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    cs[e] = make_float2(fmaf(cs[e].x, step[e].x, -cs[e].y * step[e].y), fmaf(cs[e].y, step[e].x, cs[e].x * step[e].y));
}

template <typename T, typename TOut = __half>
__device__ __forceinline__ void rope_pairs8(uint4& lo, uint4& hi, const float2* __restrict__ cs) {
  float2 c[8];
  rope_load8(c, cs);
  rope_rotate8<T, TOut>(lo, hi, c);
}

// Decode phase with RoPE: warps 1..3 (idle otherwise) walk the producer's
// stage sequence, rotate every landed K stage in shared memory (task = one
// token and one 8-dim chunk of each half; the rotated keys are fp16) and
// release it to the consumers on rot[]; the consumers wait on rot[] instead
// of full[] and read the keys as fp16.  Tokens past the
// chunk end are left alone (they are masked, and their positions may lie
// past the table).
template <typename T>
__device__ void rope_decode(const RunParams& p, RunSmem& sm, int32_t item_begin, int32_t item_end, int32_t off_items,
                            const Variant& var) {
  const int rt = threadIdx.x - 32;  // 0..95
  const int lane = threadIdx.x & 31;
  // thread = (8-frequency chunk c, token group g): tokens g, g+12, g+24, ...
  // of each stage, one walk with stride 12 per stage
  constexpr int kGroups = 12;
  const int c = rt & 7, g = rt >> 3;
  float2 step[8];
  rope_load8(step, var.rope_table + kGroups * FI_ROPE_PAIRS + 8 * c);
  __half2 amax = __float2half2_rn(0.f);
  uint32_t it = 0;
  for (int32_t i = item_begin; i < item_end; ++i) {
    const Item item = load_item(p.iws, off_items, i);
    const int nrows = item.row1 - item.row0;
    const int passes = (nrows + kRowsPerPass - 1) / kRowsPerPass;
    const int nst = (item.kv1 - item.kv0 + kStageTokens - 1) / kStageTokens;
    for (int pass = 0; pass < passes; ++pass) {
      for (int st = 0; st < nst; ++st, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        const int j0 = item.kv0 + st * kStageTokens;
        float2 cs[8];
        if (j0 + g < item.kv1) rope_load8(cs, var.rope_table + int64_t(j0 + g) * FI_ROPE_PAIRS + 8 * c);
        if (!warp_wait(&sm.full[s], ph, &sm.abort)) continue;
        // two tokens of the walk per iteration (independent loads and math)
        for (int tok = g; tok < kStageTokens && j0 + tok < item.kv1; tok += 2 * kGroups) {
          const int tok2 = tok + kGroups;
          const bool second = tok2 < kStageTokens && j0 + tok2 < item.kv1;
          float2 cs2[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) cs2[e] = cs[e];
          rope_advance8(cs2, step);
          uint4* plo = reinterpret_cast<uint4*>(&sm.dec.k[s][tok][8 * c]);
          uint4* phi = reinterpret_cast<uint4*>(&sm.dec.k[s][tok][64 + 8 * c]);
          uint4* plo2 = reinterpret_cast<uint4*>(&sm.dec.k[s][second ? tok2 : tok][8 * c]);
          uint4* phi2 = reinterpret_cast<uint4*>(&sm.dec.k[s][second ? tok2 : tok][64 + 8 * c]);
          uint4 lo = *plo, hi = *phi, lo2 = *plo2, hi2 = *phi2;
          rope_rotate8<T>(lo, hi, cs);
          if (second) rope_rotate8<T>(lo2, hi2, cs2);
          absmax_f16x8(amax, lo);
          absmax_f16x8(amax, hi);
          if (second) {
            absmax_f16x8(amax, lo2);
            absmax_f16x8(amax, hi2);
          }
          *plo = lo;
          *phi = hi;
          if (second) {
            *plo2 = lo2;
            *phi2 = hi2;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) cs[e] = cs2[e];
          rope_advance8(cs, step);
        }
        fence_proxy_async_smem();  // before the stage's next TMA write
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rot[s]);
      }
    }
  }
  if (f16x2_has_inf(amax)) atomicOr(p.iws + FI_H_STATUS, kStatusRange);
}

// One pass of up to kRowsPerPass packed rows of an item: load the rows'
// queries, stream the item's KV stages through the ring (advancing the ring
// counter it, returned), combine the half-warps' states and write O and LSE
// or the partial state.
template <typename T, bool kCap, bool kMask, bool kRope>
__device__ __forceinline__ uint32_t consume_pass(const RunParams& p, RunSmem& sm, const Item& item, int pass,
                                                 uint32_t it, int causal, int32_t num_shared, const Variant& var) {
  const int cw = (threadIdx.x >> 5) - kFirstConsumerWarp;  // consumer warp 0..7
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int L = lane & 15;
  const int hwid = cw * 2 + half;
  const int my_row = L >> 2;  // row of the group whose full score this lane holds
  const int ct = cw * 32 + lane;  // consumer thread 0..255
  const int G = p.group;
  const Request& rq = item.rq;
  const int nrows = item.row1 - item.row0;
  // a multi-head item: H KV heads, rows all of query token 0; its stages
  // hold kStageTokens / H tokens of H rows each
  const int H = item.heads;
  const int nst = ((item.kv1 - item.kv0) * H + kStageTokens - 1) >> kLog2StageTokens;
  const bool causal_i = causal && item.b >= num_shared;  // a shared block's keys are all visible

  const int prow0 = pass * kRowsPerPass;
  const int prows = min(kRowsPerPass, nrows - prow0);
  const int ng = groups_in_pass(prows);
  const int wpg = kConsumerWarps / ng;
  const int g = cw % ng;
  const int slice = cw / ng;
  const int nhw = 2 * wpg;             // half-warps sharing this row group
  const int hw = slice * 2 + half;     // index among them
  // Stage rows this half-warp scores: rb, rb + rs, ...  A multi-head
  // stage is token-major (row = token * H + head offset) and the group's
  // 4 rows share one head (G is a multiple of 4 there), hsel
  // (g * 4 / G with H = 32 / G, and 0 for a one-head item: g < 8)
  const int hsel = (g * H) >> 3;
  const int rb = hw * H + hsel, rs = nhw * H;

  // Query rows of this group, pre-scaled by scale*log2(e), as dim pairs
  // for the packed fp32 FMA (dims 2i, 2i+1 of this lane's 8).
  float2 q[kRowsPerGroup][4];
  int lim_mine = -1, lo_mine = 0;  // this lane's row: visible keys [lo, lim] (and the sink)
  // The group's row loads go out together, before any of them is used
  // (inside the per-row branch below they were issued one after another).
  uint4 qraw[kRowsPerGroup];
#pragma unroll
  for (int r = 0; r < kRowsPerGroup; ++r) {
    const int prow = prow0 + g * kRowsPerGroup + r;
    const int row = item.row0 + (prow < nrows ? prow : 0);
    const int t = row_token(item, row, G);
    const int head = item.hk * G + (row - t * G);
    qraw[r] = __ldg(reinterpret_cast<const uint4*>(p.q + int64_t(rq.qo_start + t) * p.q_stride_tok +
                                                   int64_t(head) * p.q_stride_head + L * 8));
  }
#pragma unroll
  for (int r = 0; r < kRowsPerGroup; ++r) {
    const int prow = prow0 + g * kRowsPerGroup + r;
    int lim = -1;
    if (prow < nrows) {
      const int row = item.row0 + prow;
      const int t = row_token(item, row, G);
      unpack4x2<T>(qraw[r], q[r]);
#pragma unroll
      for (int c = 0; c < 4; ++c) q[r][c] = make_float2(q[r][c].x * p.scale_log2, q[r][c].y * p.scale_log2);
      lim = causal_i ? rq.kv_len - rq.qo_len + t : rq.kv_len - 1;
      if (kMask && r == my_row) lo_mine = window_low(var, rq.kv_len - rq.qo_len + t);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) q[r][c] = make_float2(0.f, 0.f);
    }
    if (r == my_row) lim_mine = lim;
  }
  if (kRope) {
    // Rotate the query rows: this lane holds dims 8L..8L+7, the lane L^8
    // of the same half-warp the other member of each pair.
    const int f0 = (L & 7) * 8;
    const float sgn = L < 8 ? -1.f : 1.f;
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) {
      float2 pq[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        pq[c] = make_float2(__shfl_xor_sync(0xffffffffu, q[r][c].x, 8), __shfl_xor_sync(0xffffffffu, q[r][c].y, 8));
      const int prow = prow0 + g * kRowsPerGroup + r;
      if (prow < nrows) {
        const int t = row_token(item, item.row0 + prow, G);
        const float4* cs = reinterpret_cast<const float4*>(
            var.rope_table + int64_t(rq.kv_len - rq.qo_len + t) * FI_ROPE_PAIRS + f0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 w = __ldg(cs + c);  // (cos, sin) of dims 2c and 2c+1 of the lane
          q[r][c] = make_float2(fmaf(q[r][c].x, w.x, sgn * pq[c].x * w.y), fmaf(q[r][c].y, w.z, sgn * pq[c].y * w.w));
        }
      }
    }
  }
  // Visibility in stage rows: row tok * H + hsel of the stage at key j0
  // holds key j0 + tok.  It is visible to this lane's row iff row <= vhi;
  // with a window iff (unsigned)(row - vlo) < vis_cnt (one range
  // compare) or row < vsink.  Every bound is clipped to the row's last
  // visible key in the chunk, so neither a stage running past the chunk
  // nor a sink longer than the chunk or than the row's causal range
  // brings in a key the row does not see; all three move down by
  // kStageTokens rows per stage.
  const int hi_mine = min(lim_mine, item.kv1 - 1);
  const int lo_c = max(lo_mine, item.kv0) - item.kv0;  // keys before the chunk are not in any stage
  int vhi = max(hi_mine - item.kv0, -1) * H + hsel;
  int vlo = lo_c * H + hsel;
  int vsink = max(min(var.sink, hi_mine + 1) - item.kv0, 0) * H + hsel;
  const unsigned vis_cnt = kMask ? unsigned(max(0, hi_mine + 1 - item.kv0 - lo_c) * H) : 0u;

  float2 o[kRowsPerGroup][4];
#pragma unroll
  for (int r = 0; r < kRowsPerGroup; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[r][c] = make_float2(0.f, 0.f);
  float m = -INFINITY, l = 0.f;

  const int nblk = kStageTokens / (rs * kTokBlock);
  for (int st = 0; st < nst; ++st, ++it) {
    const int s = it % kStages;
    const uint32_t ph = (it / kStages) & 1;
    // warp-uniform result: the body below shuffles across the warp
    if (warp_wait(kRope ? &sm.rot[s] : &sm.full[s], ph, &sm.abort)) {
      for (int blk = 0; blk < nblk; ++blk) {
        float sc[kTokBlock];
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) {
          const int tok = rb + (blk * kTokBlock + u) * rs;  // stage row
          const uint4 kv = *reinterpret_cast<const uint4*>(&sm.dec.k[s][tok][L * 8]);
          float2 f[4];
          unpack4x2<std::conditional_t<kRope, __half, T>>(kv, f);  // rotated keys are fp16
          float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            a0 = fma2(q[0][c], f[c], a0);
            a1 = fma2(q[1][c], f[c], a1);
            a2 = fma2(q[2][c], f[c], a2);
            a3 = fma2(q[3][c], f[c], a3);
          }
          float sfull = reduce_rows4(a0.x + a0.y, a1.x + a1.y, a2.x + a2.y, a3.x + a3.y, L);
          if (kCap) sfull = soft_cap_log2(sfull, var.cap_a, var.cap_b);
          const bool seen = kMask ? (unsigned(tok - vlo) < vis_cnt || tok < vsink) : tok <= vhi;
          sc[u] = seen ? sfull : -INFINITY;
        }
        float mt[kTokBlock];  // pairwise (tree) maximum of the block's logits
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) mt[u] = sc[u];
#pragma unroll
        for (int w = kTokBlock / 2; w > 0; w >>= 1)
#pragma unroll
          for (int u = 0; u < w; ++u) mt[u] = fmaxf(mt[u], mt[u + w]);
        const float mx = mt[0];
        float m_new = m;
        if (mx > m + kLazyRescale) m_new = mx;  // also taken on the first visible key (m = -inf)
        const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);
        float ps[kTokBlock];
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) {
          ps[u] = (m_new == -INFINITY) ? 0.f : ex2(sc[u] - m_new);
          psum += ps[u];
        }
        l = l * alpha + psum;
        m = m_new;
        float* x = reinterpret_cast<float*>(sm.dec.xch[hwid]);
        if ((L & 3) == 0) {
#pragma unroll
          for (int u = 0; u < kTokBlock; ++u) x[u * 4 + my_row] = ps[u];
          x[kTokBlock * 4 + my_row] = alpha;
        }
        __syncwarp();
        const float4 al = sm.dec.xch[hwid][kTokBlock];
        if (__any_sync(0xffffffffu, al.x != 1.f || al.y != 1.f || al.z != 1.f || al.w != 1.f)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            o[0][c] = make_float2(o[0][c].x * al.x, o[0][c].y * al.x);
            o[1][c] = make_float2(o[1][c].x * al.y, o[1][c].y * al.y);
            o[2][c] = make_float2(o[2][c].x * al.z, o[2][c].y * al.z);
            o[3][c] = make_float2(o[3][c].x * al.w, o[3][c].y * al.w);
          }
        }
#pragma unroll
        for (int u = 0; u < kTokBlock; ++u) {
          const int tok = rb + (blk * kTokBlock + u) * rs;
          const float4 pu = sm.dec.xch[hwid][u];
          const uint4 vv = *reinterpret_cast<const uint4*>(&sm.dec.v[s][tok][L * 8]);
          float2 f[4];
          unpack4x2<T>(vv, f);
          const float2 p0 = make_float2(pu.x, pu.x), p1 = make_float2(pu.y, pu.y);
          const float2 p2 = make_float2(pu.z, pu.z), p3 = make_float2(pu.w, pu.w);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            o[0][c] = fma2(p0, f[c], o[0][c]);
            o[1][c] = fma2(p1, f[c], o[1][c]);
            o[2][c] = fma2(p2, f[c], o[2][c]);
            o[3][c] = fma2(p3, f[c], o[3][c]);
          }
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    vhi -= kStageTokens;
    vlo -= kStageTokens;
    vsink -= kStageTokens;
  }

  // Eight row groups (a pass of more than 16 rows): each warp holds one
  // group, its two half-warps the same 4 rows over different tokens.  Their
  // states merge by shuffles, half-warp 0's first, and half-warp h writes
  // rows 2h and 2h + 1; no shared memory and no barrier.
  if (ng == kGroupsPerPass) {
    float w0[kRowsPerGroup], w1[kRowsPerGroup], Mr[kRowsPerGroup], Lr[kRowsPerGroup];
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) {
      const float m0 = __shfl_sync(0xffffffffu, m, r * 4), m1 = __shfl_sync(0xffffffffu, m, 16 + r * 4);
      const float l0 = __shfl_sync(0xffffffffu, l, r * 4), l1 = __shfl_sync(0xffffffffu, l, 16 + r * 4);
      Mr[r] = fmaxf(m0, m1);
      w0[r] = m0 == -INFINITY ? 0.f : ex2(m0 - Mr[r]);
      w1[r] = m1 == -INFINITY ? 0.f : ex2(m1 - Mr[r]);
      Lr[r] = w0[r] * l0 + w1[r] * l1;
    }
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) {
      const float inv = Lr[r] > 0.f ? 1.f / Lr[r] : 0.f;
      float v[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 x = o[r][c];
        const float2 y = make_float2(__shfl_xor_sync(0xffffffffu, x.x, 16), __shfl_xor_sync(0xffffffffu, x.y, 16));
        const float2 a = half ? y : x, b = half ? x : y;  // half-warp 0's state first in both halves
        v[2 * c] = (a.x * w0[r] + b.x * w1[r]) * inv;
        v[2 * c + 1] = (a.y * w0[r] + b.y * w1[r]) * inv;
      }
      const int prow = prow0 + g * kRowsPerGroup + r;
      if ((r >> 1) != half || prow >= nrows) continue;
      const float lse_v = Lr[r] > 0.f ? (Mr[r] + __log2f(Lr[r])) * 0.69314718055994531f : -INFINITY;
      if (item.part < 0) {
        const int row = item.row0 + prow;
        const int t = row_token(item, row, G);
        const int head = item.hk * G + (row - t * G);
        const int64_t tok = rq.qo_start + t;
        uint4 packed;
        packed.x = Elem<T>::from_float2(v[0], v[1]);
        packed.y = Elem<T>::from_float2(v[2], v[3]);
        packed.z = Elem<T>::from_float2(v[4], v[5]);
        packed.w = Elem<T>::from_float2(v[6], v[7]);
        *reinterpret_cast<uint4*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + L * 8) = packed;
        if (L == 0 && p.lse) p.lse[tok * p.num_qo_heads + head] = lse_v;
      } else {
        const int64_t prw = int64_t(item.part) + prow;
        float4* dst = reinterpret_cast<float4*>(p.fws + p.partial_o_offset + prw * kHeadDim + L * 8);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        if (L == 0) p.fws[prw] = lse_v;
      }
    }
    return it;
  }

  // This half-warp's state -> shared memory, then merge per row (comb_o
  // shares its bytes with the exchange buffers of the stage loop).
  named_barrier_sync(1, 32 * kConsumerWarps);
#pragma unroll
  for (int r = 0; r < kRowsPerGroup; ++r) {
    float4* dst = reinterpret_cast<float4*>(&sm.dec.comb_o[hwid][r][L * 8]);
    dst[0] = make_float4(o[r][0].x, o[r][0].y, o[r][1].x, o[r][1].y);
    dst[1] = make_float4(o[r][2].x, o[r][2].y, o[r][3].x, o[r][3].y);
  }
  if ((L & 3) == 0) {
    sm.dec.comb_m[hwid][my_row] = m;
    sm.dec.comb_l[hwid][my_row] = l;
  }
  named_barrier_sync(1, 32 * kConsumerWarps);
  if (!sm.abort) {
    for (int task = ct; task < prows * 32; task += 32 * kConsumerWarps) {
      const int pr = task >> 5, ch = task & 31;
      const int gg = pr / kRowsPerGroup, r = pr % kRowsPerGroup;
      float M = -INFINITY;
      for (int sl = 0; sl < wpg; ++sl)
        for (int h2 = 0; h2 < 2; ++h2) M = fmaxf(M, sm.dec.comb_m[(gg + sl * ng) * 2 + h2][r]);
      float Ls = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
        for (int sl = 0; sl < wpg; ++sl)
          for (int h2 = 0; h2 < 2; ++h2) {
            const int id = (gg + sl * ng) * 2 + h2;
            const float w = ex2(sm.dec.comb_m[id][r] - M);
            Ls += w * sm.dec.comb_l[id][r];
            const float4 v = *reinterpret_cast<const float4*>(&sm.dec.comb_o[id][r][ch * 4]);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
          }
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      const float lse_v = Ls > 0.f ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
      const int prow = prow0 + pr;
      if (item.part < 0) {
        const int row = item.row0 + prow;
        const int t = row_token(item, row, G);
        const int head = item.hk * G + (row - t * G);
        const int64_t tok = rq.qo_start + t;
        uint2 packed;
        packed.x = Elem<T>::from_float2(acc.x, acc.y);
        packed.y = Elem<T>::from_float2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.o + tok * p.o_stride_tok + int64_t(head) * p.o_stride_head + ch * 4) =
            packed;
        if (ch == 0 && p.lse) p.lse[tok * p.num_qo_heads + head] = lse_v;
      } else {
        const int64_t prw = int64_t(item.part) + prow;
        *reinterpret_cast<float4*>(p.fws + p.partial_o_offset + prw * kHeadDim + ch * 4) = acc;
        if (ch == 0) p.fws[prw] = lse_v;
      }
    }
  }
  named_barrier_sync(1, 32 * kConsumerWarps);
  return it;
}

template <typename T, bool kCap, bool kMask, bool kRope>
__device__ void consume(const RunParams& p, RunSmem& sm, int32_t item_begin, int32_t item_end, int32_t off_items,
                        int32_t off_req, int32_t off_merge, int32_t off_cnt, int causal, int32_t num_shared,
                        const Variant var) {
  const int ct = threadIdx.x - 32 * kFirstConsumerWarp;  // consumer thread 0..255
  uint32_t it = 0;

  // Items in the order dealt; each pass of an item loads its query rows,
  // streams the item's KV stages and combines the half-warps' states.
  // (Loading the next item's descriptor a whole item ahead, its query rows
  // before this item's combine, or splitting the combine's loop over the
  // idle lanes, measured slower on some of the workloads: the added live
  // registers spill, which costs more than the latency saved.)
  for (int32_t i = item_begin; i < item_end; ++i) {
    const Item item = load_item(p.iws, off_items, i);
    const int passes = (item.row1 - item.row0 + kRowsPerPass - 1) / kRowsPerPass;
    for (int pass = 0; pass < passes; ++pass)
      it = consume_pass<T, kCap, kMask, kRope>(p, sm, item, pass, it, causal, num_shared, var);
    if (item.merge >= 0)
      merge_split_unit<T>(p, item, item.rq, off_merge, off_cnt, ct, 32 * kConsumerWarps, 1, &sm.merge_last,
                          sm.abort);
  }
}

}  // namespace fi

#include "prefill_kernel.cuh"

namespace fi {

// ---------------------------------------------------------------- kernel

// A CTA's items come prefill-class (256-row tiles) first, then decode-class
// (16-row tiles); returns the index of its first item for the CUDA-core path:
// a decode-class item, or a prefill-class item whose KV cache has no
// tensor-core maps (pages under 8 tokens, or G not dividing 128).  The
// tensor-core phase takes the items before it.  Called by whole warps: lane
// l looks at item i0 + l (its request's row count decides the class), so 32
// items cost one load.
__device__ __forceinline__ int32_t first_cuda_core_item(const RunParams& p, int32_t begin, int32_t end,
                                                        int32_t off_items, int32_t off_req, int32_t num_shared) {
  const int lane = threadIdx.x & 31;
  for (int32_t i0 = begin; i0 < end; i0 += 32) {
    bool cc = true;  // past the CTA's last item counts as the boundary
    if (i0 + lane < end) {
      const int32_t* it = p.iws + off_items + FI_ITEM_INTS * (i0 + lane);
      const int32_t b = __ldg(it), qo_len = __ldg(it + 9);  // the item's own copy of its request's qo_len
      cc = qo_len * p.group <= FI_TILE_DECODE || !cache_of(p, b, num_shared).tc;
    }
    const unsigned m = __ballot_sync(0xffffffffu, cc);
    if (m) return min(end, i0 + __ffs(m) - 1);
  }
  return end;
}

template <typename T, bool kCap, bool kMask, bool kRope>
__global__ void __launch_bounds__(kThreads, 1) paged_attention_kernel(const __grid_constant__ RunParams p) {
  // Casting the __shared__ array itself keeps every access below in the
  // shared address space (LDS/STS rather than generic loads).  The swizzled
  // TMA/MMA operand blocks need a 1024-byte aligned base; it is checked, and
  // a misaligned base is reported instead of being used.
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  RunSmem& sm = *reinterpret_cast<RunSmem*>(smem_raw);
  // A merge launched behind this run may be scheduled from now on: its blocks
  // take SMs as this grid's CTAs leave and wait for the grid to complete.
  if (threadIdx.x == 0) let_dependents_start();
  const int32_t* iws = p.iws;
  const int32_t magic = ws_header(iws, FI_H_MAGIC);
  const int32_t n_items = ws_header(iws, FI_H_NUM_ITEMS);
  const int32_t n_ctas = ws_header(iws, FI_H_NUM_CTAS);
  const int32_t off_cta = ws_header(iws, FI_H_OFF_CTA);
  // The plan in the workspace must also fit the buffers of this launch: its
  // partial rows the float workspace, its query tokens Q and O, its head
  // counts and page size the tensor maps.  A workspace re-planned after the
  // arguments were checked on the host is refused here, before any write.
  // (The header fields share one cache line; their loads go out together.)
  const int32_t h_rows = ws_header(iws, FI_H_PARTIAL_ROWS), h_qo = ws_header(iws, FI_H_TOTAL_QO);
  const int32_t h_hq = ws_header(iws, FI_H_NUM_QO_HEADS), h_hkv = ws_header(iws, FI_H_NUM_KV_HEADS);
  const int32_t h_page = ws_header(iws, FI_H_PAGE_SIZE);
  const int32_t num_shared = ws_header(iws, FI_H_NUM_SHARED), h_spage = ws_header(iws, FI_H_SHARED_PAGE_SIZE);
  // A RoPE plan runs on the RoPE instantiation, or -- its operands rotated by
  // a pass before the run -- on the plain one when every item is a
  // tensor-core item (the CUDA-core path would read unrotated keys); a plan
  // without RoPE runs on the plain instantiation only.
  const int32_t h_dec = ws_header(iws, FI_H_NUM_DECODE_ITEMS);
  const bool h_rope = ws_header(iws, FI_H_ROPE_MAX_POS) > 0;
  bool bad = magic != FI_PLAN_MAGIC || n_ctas != int32_t(gridDim.x) || (smem_u32(smem_raw) & 1023u) != 0 ||
             h_rows < 0 || h_rows > p.max_partial_rows || h_qo < 0 || h_qo > p.q_num_tokens ||
             h_hq != p.num_qo_heads || h_hkv != p.num_kv_heads || h_page != p.kv[0].page_size ||
             num_shared < 0 || (num_shared > 0 && (!p.has_shared || h_spage != p.kv[1].page_size)) ||
             (kRope ? !h_rope : h_rope && !(p.qk_prerotated && h_dec == 0));
  int32_t begin = 0, end = 0;
  if (!bad) {
    begin = __ldg(iws + off_cta + blockIdx.x);
    end = __ldg(iws + off_cta + blockIdx.x + 1);
    bad = begin < 0 || end < begin || end > n_items;
  }
  if (bad) {
    if (threadIdx.x == 0) atomicOr(p.iws + FI_H_STATUS, kStatusBadPlan);
    return;
  }
  const int32_t off_items = ws_header(iws, FI_H_OFF_ITEMS);
  const int32_t off_req = ws_header(iws, FI_H_OFF_REQUESTS);
  const int32_t off_merge = ws_header(iws, FI_H_OFF_MERGE);
  const int32_t off_cnt = ws_header(iws, FI_H_OFF_COUNTERS);
  const int causal = ws_header(iws, FI_H_CAUSAL);
  Variant var;
  var.window_left = ws_header(iws, FI_H_WINDOW_LEFT);
  var.sink = ws_header(iws, FI_H_SINK_TOKENS);
  const float cap = __int_as_float(ws_header(iws, FI_H_SOFT_CAP_BITS));
  var.cap_a = cap * 1.4426950408889634f;
  var.cap_b = cap > 0.f ? 2.f / cap : 0.f;
  var.rope_table = kRope ? reinterpret_cast<const float2*>(iws + ws_header(iws, FI_H_ROPE_TABLE_OFF)) : nullptr;
  const int warp = threadIdx.x >> 5;
  const int32_t mid = first_cuda_core_item(p, begin, end, off_items, off_req, num_shared);
  const bool tc_phase = mid > begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);               // the producer's arrive.expect_tx; TMA completes the bytes
      mbar_init(&sm.empty[s], kConsumerWarps); // one arrival per consumer warp
    }
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.q_rot, 2);
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.rot[s], 3);  // warps 1..3
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.o_ready[s], 1);
      mbar_init(&sm.k_rot[s], 2);  // the two rotation warps
      mbar_init(&sm.p_full[s][0], 4);  // one arrival per warp of the M tile's softmax warpgroup
      mbar_init(&sm.p_full[s][1], 4);
      mbar_init(&sm.o_free[s], 4);
    }
    sm.abort = 0;
    sm.merge_last = 0;
    sm.merge_last_pf = 0;
    fence_mbar_init();
  }
  if (tc_phase && warp == kMmaWarp) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  if (tc_phase) {
    // Each branch returns to kRegsLaunch before the code paths merge: the
    // softmax warpgroups release their registers before the phase barrier,
    // the loader warpgroup takes its share back after it.
    if (warp < kSoftmaxWarp0) {
      tc::setmaxnreg_dec<kRegsLoader>();
      // With RoPE, warps 2 and 3 rotate Q and K tiles in shared memory and
      // warp 0 loads all three operands -- unless a pass before the run has
      // rotated them (then the plain roles, fp16 Q and K; a plan with no
      // CUDA-core item then runs on the instantiation without RoPE)
      const bool rot_roles = kRope && !p.qk_prerotated;
      if (warp == 0) {
        if (rot_roles)
          pf_produce<kProduceQKV>(p, sm, begin, mid, off_items, off_req, num_shared);
        else
          pf_produce<kProduceQK>(p, sm, begin, mid, off_items, off_req, num_shared);
      } else if (warp == kMmaWarp) {
        pf_mma<T, kRope>(p, sm, begin, mid, off_items);
        __syncwarp();
      } else if (rot_roles) {
        pf_rope<T>(p, sm, begin, mid, off_items, off_req, var);  // warps 2 and 3
      } else if (warp == kVWarp) {
        pf_produce<kProduceV>(p, sm, begin, mid, off_items, off_req, num_shared);
      }
      tc::fence_before_sync();
      named_barrier_sync_unaligned(kPhaseBarrier, kThreads);
      tc::fence_after_sync();
      tc::setmaxnreg_inc<kRegsLaunch>();
    } else {
      tc::setmaxnreg_inc<kRegsSoftmax>();
      pf_softmax<T, kCap, kMask>(p, sm, begin, mid, off_items, off_req, off_merge, off_cnt, causal, num_shared,
                                 var);
      tc::setmaxnreg_dec<kRegsLaunch>();
      tc::fence_before_sync();
      named_barrier_sync_unaligned(kPhaseBarrier, kThreads);
      tc::fence_after_sync();
    }
  }

  if (warp == 0) {
    produce(p, sm, mid, end, off_items, off_req, num_shared);
  } else if (warp >= kFirstConsumerWarp) {
    consume<T, kCap, kMask, kRope>(p, sm, mid, end, off_items, off_req, off_merge, off_cnt, causal, num_shared, var);
  } else if (kRope && warp >= 1 && warp <= 3) {
    rope_decode<T>(p, sm, mid, end, off_items, var);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tc_phase && warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(sm.tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(p.iws + FI_H_STATUS, sm.abort);
}

}  // namespace fi
