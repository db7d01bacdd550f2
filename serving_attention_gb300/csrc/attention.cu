// attention.cu -- C-ABI entry points of the run kernel, the state merge
// kernel, the default plan config and the device status query.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fi.h"
#include "attention_kernel.cuh"
#include "launch.h"
#include "workspace.h"

namespace fi {

// ------------------------------------------------------------ merge kernel

// Storage <-> fp32 for 8 consecutive elements.
template <typename T>
struct Vec8 {
  __device__ __forceinline__ static void load(const T* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const float2 a = Elem<T>::to_float2(u.x), b = Elem<T>::to_float2(u.y);
    const float2 c = Elem<T>::to_float2(u.z), d = Elem<T>::to_float2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ __forceinline__ static void store(T* p, const float (&f)[8]) {
    uint4 u;
    u.x = Elem<T>::from_float2(f[0], f[1]);
    u.y = Elem<T>::from_float2(f[2], f[3]);
    u.z = Elem<T>::from_float2(f[4], f[5]);
    u.w = Elem<T>::from_float2(f[6], f[7]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};

template <>
struct Vec8<float> {
  __device__ __forceinline__ static void load(const float* p, float (&f)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  __device__ __forceinline__ static void store(float* p, const float (&f)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
};

// One (row, head) state per 16 threads, 8 elements per thread (head_dim 128).
// Every thread of a state reads both inputs before any thread writes, so the
// output may alias either input.
template <typename T>
__global__ void __launch_bounds__(256) merge_states_kernel(const T* __restrict__ va, const float* sa, const T* vb,
                                                            const float* sb, T* vo, float* so, int64_t states) {
  const int64_t st = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int part = threadIdx.x & 15;
  if (st >= states) return;
  const float la = sa[st] * 1.4426950408889634f;  // natural log -> log2
  const float lb = sb[st] * 1.4426950408889634f;
  float a[8], b[8], r[8];
  Vec8<T>::load(va + st * kHeadDim + part * 8, a);
  Vec8<T>::load(vb + st * kHeadDim + part * 8, b);
  float lse;
  if (la == -INFINITY && lb == -INFINITY) {
#pragma unroll
    for (int c = 0; c < 8; ++c) r[c] = 0.f;
    lse = -INFINITY;
  } else {
    const float mx = fmaxf(la, lb);
    const float wa = ex2(la - mx), wb = ex2(lb - mx);
    const float inv = 1.f / (wa + wb);
#pragma unroll
    for (int c = 0; c < 8; ++c) r[c] = (wa * a[c] + wb * b[c]) * inv;
    lse = (mx + __log2f(wa + wb)) * 0.69314718055994531f;
  }
  __syncwarp();
  Vec8<T>::store(vo + st * kHeadDim + part * 8, r);
  if (part == 0) so[st] = lse;
}

// Late merge of split units (those the plan marks late: prefill-class
// tiles), launched after the run on the same stream.  Tasks are (merge unit,
// packed row) pairs, unit-major, walked by every warp of a fixed grid with a
// grid stride, and the counts come from the workspace header, so a graph
// captured once replays correctly for any later plan.  Lane l holds dims
// 4l..4l+3.  The arithmetic and the chunk order of the sums are those of the
// in-run merge, so a unit's result does not depend on which of the two
// merged it.
// Nothing is merged when the status word reports an error (the partial
// states may be incomplete).
template <typename T>
__global__ void __launch_bounds__(256) late_merge_kernel(const int32_t* __restrict__ iws,
                                                         const float* __restrict__ fws, int64_t partial_o_offset,
                                                         T* o, int64_t o_stride_tok, int64_t o_stride_head,
                                                         float* lse, int num_qo_heads, int group) {
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();  // launched early behind the run: its partial rows are written from here on
  if (iws[FI_H_STATUS] != 0 || iws[FI_H_NUM_LATE_MERGE] == 0) return;
  const int64_t tasks = int64_t(iws[FI_H_NUM_MERGE]) * FI_TILE_PREFILL;
  const int32_t* merge = iws + iws[FI_H_OFF_MERGE];
  const int32_t* reqs = iws + iws[FI_H_OFF_REQUESTS];
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t task = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); task < tasks; task += warps) {
    const int32_t* mu = merge + FI_MERGE_INTS * (task / FI_TILE_PREFILL);
    const int pr = int(task % FI_TILE_PREFILL);
    const int row0 = mu[2], nrows = mu[3] - row0;
    if (!mu[FI_MERGE_LATE] || pr >= nrows) continue;
    const int n = mu[4];
    const int64_t base = mu[5];
    const float* part_lse = fws + base + pr;  // chunk c at [c * nrows]
    const float4* part_o = reinterpret_cast<const float4*>(fws + partial_o_offset + (base + pr) * kHeadDim) + lane;
    const int64_t o_step = int64_t(nrows) * (kHeadDim / 4);  // float4s from chunk c to c + 1
    // groups of 32 chunks: lane c holds chunk c's LSE, the group's max comes
    // from a butterfly, and the partial rows are loaded 8 at a time ahead of
    // their use; the weights and sums still run in chunk order
    float M = -INFINITY;
    for (int c0 = 0; c0 < n; c0 += 32)
      M = fmaxf(M, c0 + lane < n ? __ldcg(part_lse + int64_t(c0 + lane) * nrows) : -INFINITY);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int c0 = 0; c0 < n; c0 += 32) {
        const float w_mine =
            c0 + lane < n ? ex2((__ldcg(part_lse + int64_t(c0 + lane) * nrows) - M) * 1.4426950408889634f) : 0.f;
        const int cn = min(32, n - c0);
        for (int g0 = 0; g0 < cn; g0 += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (g0 + u < cn) v[u] = __ldcg(part_o + int64_t(c0 + g0 + u) * o_step);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float w = __shfl_sync(0xffffffffu, w_mine, (g0 + u) & 31);
            if (g0 + u < cn) {
              Ls += w;
              acc.x += w * v[u].x;
              acc.y += w * v[u].y;
              acc.z += w * v[u].z;
              acc.w += w * v[u].w;
            }
          }
        }
      }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    const int row = row0 + pr;
    const int t = row / group;
    const int head = mu[1] * group + (row - t * group);
    const int64_t tok = int64_t(reqs[FI_REQ_INTS * mu[0]]) + t;
    uint2 packed;
    packed.x = Elem<T>::from_float2(acc.x * inv, acc.y * inv);
    packed.y = Elem<T>::from_float2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(o + tok * o_stride_tok + int64_t(head) * o_stride_head + lane * 4) = packed;
    if (lane == 0 && lse) lse[tok * num_qo_heads + head] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
  }
}

template <typename T>
cudaError_t launch_late_merge(const RunParams& p, int32_t blocks, cudaStream_t s) {
  return launch_behind_run(late_merge_kernel<T>, blocks, 256, s, static_cast<const int32_t*>(p.iws),
                           static_cast<const float*>(p.fws), p.partial_o_offset, reinterpret_cast<T*>(p.o),
                           p.o_stride_tok, p.o_stride_head, p.lse, int(p.num_qo_heads), int(p.group));
}

// RoPE table: (cos, sin) of (pos / scale) * theta^(-2i/128) for pos <
// max_pos, i < 64, computed in fp64 and rounded once to fp32.
__global__ void rope_table_kernel(float2* table, int64_t entries, double theta, double inv_scale) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= entries) return;
  const int64_t pos = idx / FI_ROPE_PAIRS;
  const int i = int(idx % FI_ROPE_PAIRS);
  const double freq = pow(theta, -2.0 * i / double(2 * FI_ROPE_PAIRS));
  double sn, cs;
  sincos(double(pos) * inv_scale * freq, &sn, &cs);
  table[idx] = make_float2(float(cs), float(sn));
}

// Rotation passes outside attention -- the standalone forms and the pass of
// the pre-rotated run -- flat over the requests they rotate, so that one
// long request is spread over the whole grid.  Each CTA first lists those
// requests (for the pre-rotated run only prefill-class ones) with prefix sums
// of their pages and query tokens in shared memory; past kRopeListCap
// requests it walks the whole request table instead, skipping row by row.
// Unit u < nk covers 32 consecutive key slots of the listed requests' pages,
// unit u >= nk 32 of their query tokens; key j of a request sits at position
// j, its query token t at kv_len - qo_len + t.  Warp 0 finds the rows of a
// CTA's next unit (a binary search over the prefix sums per row) while the
// block rotates the current one.  A task is one row (slot or token, and a
// head) and one 8-dim chunk of each half; a thread issues the loads of four
// tasks before it rotates any.  The counts come from the plan in the
// workspace, so a graph captured once serves later plans.  fp16 output past
// the fp16 range (|x| > 65504, which a bf16 input can reach) records
// kStatusRange.
struct RopePass {
  int32_t* iws;
  const uint16_t* k_in;
  int64_t ki[3];
  uint16_t* k_out;
  int64_t ko[3];
  const int32_t* kv_indices;
  const uint16_t* q_in;
  int64_t qi_tok, qi_head;
  uint16_t* q_out;
  int64_t qo_tok, qo_head;
  int log2_page, num_kv_heads, num_qo_heads, group;
  int keys, queries;  // what the pass rotates
  int prefill_only;   // leave decode-class requests (at most 16 packed rows) alone
};

constexpr int kRopeUnitRows = 32, kRopeLoadsAhead = 4, kRopeThreads = 256, kRopeListCap = 1024;

template <typename T, typename TOut>
__global__ void __launch_bounds__(kRopeThreads, 3) rope_pass_kernel(const __grid_constant__ RopePass a) {
  __shared__ int32_t s_req[kRopeListCap];                      // listed request
  __shared__ int32_t s_pages[kRopeListCap + 1], s_toks[kRopeListCap + 1];  // prefix sums over the list
  __shared__ int32_t s_warp[kRopeThreads / 32], s_n;
  // per unit row, double-buffered: element offsets of the row (head 0), -1
  // when it is not rotated, and its position
  __shared__ int64_t s_in[2][kRopeUnitRows], s_out[2][kRopeUnitRows];
  __shared__ int32_t s_pos[2][kRopeUnitRows];
  const int32_t* iws = a.iws;
  const int batch = __ldg(iws + FI_H_BATCH);
  if (batch <= 0) return;
  const int32_t off_req = __ldg(iws + FI_H_OFF_REQUESTS);
  const float2* table = reinterpret_cast<const float2*>(iws + __ldg(iws + FI_H_ROPE_TABLE_OFF));
  const int P = 1 << a.log2_page;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto wanted = [&](const Request& rq) { return !(a.prefill_only && rq.qo_len * a.group <= FI_TILE_DECODE); };

  // The list: requests in table order, block-wide compaction 256 at a time.
  if (tid == 0) s_n = 0;
  __syncthreads();
  bool listed = true;
  for (int b0 = 0; b0 < batch && listed; b0 += kRopeThreads) {
    const int b = b0 + tid;
    bool take = false;
    if (b < batch) take = wanted(load_request(iws, off_req, b));
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (lane == 0) s_warp[warp] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kRopeThreads / 32; ++w) {
      before += w < warp ? s_warp[w] : 0;
      total += s_warp[w];
    }
    const int n0 = s_n;
    if (n0 + total > kRopeListCap) {
      listed = false;  // every thread sees the same counts
    } else if (take) {
      s_req[n0 + before + __popc(m & ((1u << lane) - 1u))] = b;
    }
    __syncthreads();
    if (tid == 0 && listed) s_n = n0 + total;
    __syncthreads();
  }
  const int n = listed ? s_n : batch;
  if (listed) {
    // prefix sums of pages and tokens: thread t sums entries [4t, 4t + 4)
    // of each group of 1024, then a scan of the 256 partial sums
    int carry_p = 0, carry_t = 0;
    if (tid == 0) s_pages[0] = s_toks[0] = 0;
    for (int e0 = 0; e0 < n; e0 += 4 * kRopeThreads) {
      int vp[4], vt[4], sp = 0, st = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = e0 + 4 * tid + k;
        vp[k] = vt[k] = 0;
        if (e < n) {
          const Request rq = load_request(iws, off_req, s_req[e]);
          vp[k] = a.keys ? (rq.kv_len + P - 1) >> a.log2_page : 0;
          vt[k] = a.queries ? rq.qo_len : 0;
        }
        sp += vp[k];
        st += vt[k];
      }
      int ip = sp, it = st;  // inclusive warp scan
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, ip, d), ut = __shfl_up_sync(0xffffffffu, it, d);
        if (lane >= d) {
          ip += up;
          it += ut;
        }
      }
      __syncthreads();
      if (lane == 31) {
        s_warp[warp] = ip;
        s_in[0][warp] = it;  // borrowed as scratch before the units start
      }
      __syncthreads();
      int wp = 0, wt = 0, tp = 0, tt = 0;
      for (int w = 0; w < kRopeThreads / 32; ++w) {
        wp += w < warp ? s_warp[w] : 0;
        wt += w < warp ? int(s_in[0][w]) : 0;
        tp += s_warp[w];
        tt += int(s_in[0][w]);
      }
      int rp = carry_p + wp + ip - sp, rt = carry_t + wt + it - st;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = e0 + 4 * tid + k;
        rp += vp[k];
        rt += vt[k];
        if (e < n) {
          s_pages[e + 1] = rp;
          s_toks[e + 1] = rt;
        }
      }
      carry_p += tp;
      carry_t += tt;
    }
    __syncthreads();
  }
  // Entry e of the list (or request e of the table): its request, and the
  // first page and token of its share of the flat unit space.
  auto req_of = [&](int e) { return listed ? s_req[e] : e; };
  auto first_page = [&](int e) {
    if (listed) return s_pages[e];
    if (e == batch) {
      const Request l = load_request(iws, off_req, batch - 1);
      return l.page_start + ((l.kv_len + P - 1) >> a.log2_page);
    }
    return __ldg(iws + off_req + FI_REQ_INTS * e + 2);
  };
  auto first_token = [&](int e) {
    if (listed) return s_toks[e];
    if (e == batch) {
      const Request l = load_request(iws, off_req, batch - 1);
      return l.qo_start + l.qo_len;
    }
    return __ldg(iws + off_req + FI_REQ_INTS * e);
  };
  const int64_t slots = a.keys ? int64_t(first_page(n)) << a.log2_page : 0;
  const int64_t total_qo = a.queries ? first_token(n) : 0;
  const int64_t nk = (slots + kRopeUnitRows - 1) / kRopeUnitRows;
  const int64_t nu = nk + (total_qo + kRopeUnitRows - 1) / kRopeUnitRows;
  // rows of unit u into buffer `buf` (lane = row of the unit; warp 0 only)
  auto find_rows = [&](int64_t u, int buf) {
    const bool key_unit = u < nk;
    const int64_t x = (key_unit ? u : u - nk) * kRopeUnitRows + lane;
    int64_t bi = -1, bo = -1;
    int pos = 0;
    if (x < (key_unit ? slots : total_qo)) {
      const int64_t g = key_unit ? (x >> a.log2_page) : x;  // flat page, or flat query token
      int lo = 0, hi = n - 1;  // the last entry whose first page (token) is at or before g
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((key_unit ? first_page(mid) : first_token(mid)) <= g)
          lo = mid;
        else
          hi = mid - 1;
      }
      const Request rq = load_request(iws, off_req, req_of(lo));
      if (listed || wanted(rq)) {
        if (key_unit) {
          const int slot = int(x & (P - 1));
          const int64_t pg = g - first_page(lo);  // page of the request
          const int64_t j = (pg << a.log2_page) + slot;
          if (j < rq.kv_len) {
            const int64_t page = __ldg(a.kv_indices + rq.page_start + pg);
            bi = page * a.ki[0] + slot * a.ki[1];
            bo = page * a.ko[0] + slot * a.ko[1];
            pos = int(j);
          }
        } else {
          const int64_t t = g - first_token(lo);  // token of the request
          bi = (rq.qo_start + t) * a.qi_tok;
          bo = (rq.qo_start + t) * a.qo_tok;
          pos = rq.kv_len - rq.qo_len + int(t);
        }
      }
    }
    s_in[buf][lane] = bi;
    s_out[buf][lane] = bo;
    s_pos[buf][lane] = pos;
  };
  __half2 amax = __float2half2_rn(0.f);
  int buf = 0;
  if (warp == 0 && blockIdx.x < nu) find_rows(blockIdx.x, 0);
  __syncthreads();
  for (int64_t u = blockIdx.x; u < nu; u += gridDim.x, buf ^= 1) {
    // the next unit's rows go to the other buffer, read after the barrier below
    if (warp == 0 && u + gridDim.x < nu) find_rows(u + gridDim.x, buf ^ 1);
    const bool key_unit = u < nk;
    const int H = key_unit ? a.num_kv_heads : a.num_qo_heads;
    const uint16_t* src = key_unit ? a.k_in : a.q_in;
    uint16_t* dst = key_unit ? a.k_out : a.q_out;
    const int64_t hs_in = key_unit ? a.ki[2] : a.qi_head, hs_out = key_unit ? a.ko[2] : a.qo_head;
    const int tasks = kRopeUnitRows * H * 8;
    for (int t0 = tid; t0 < tasks; t0 += kRopeLoadsAhead * kRopeThreads) {
      uint4 lo[kRopeLoadsAhead], hi[kRopeLoadsAhead];
      int64_t ob[kRopeLoadsAhead];
      const float2* cs[kRopeLoadsAhead];
#pragma unroll
      for (int k = 0; k < kRopeLoadsAhead; ++k) {
        const int t = t0 + k * kRopeThreads;
        ob[k] = -1;
        if (t < tasks) {
          const int r = t / (H * 8), rem = t - r * (H * 8);
          const int h = rem >> 3, c = rem & 7;
          const int64_t ib = s_in[buf][r];
          if (ib >= 0) {
            const int64_t i = ib + h * hs_in + 8 * c;
            lo[k] = *reinterpret_cast<const uint4*>(src + i);
            hi[k] = *reinterpret_cast<const uint4*>(src + i + 64);
            ob[k] = s_out[buf][r] + h * hs_out + 8 * c;
            cs[k] = table + int64_t(s_pos[buf][r]) * FI_ROPE_PAIRS + 8 * c;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kRopeLoadsAhead; ++k) {
        if (ob[k] < 0) continue;
        rope_pairs8<T, TOut>(lo[k], hi[k], cs[k]);
        if (std::is_same<TOut, __half>::value) {
          absmax_f16x8(amax, lo[k]);
          absmax_f16x8(amax, hi[k]);
        }
        *reinterpret_cast<uint4*>(dst + ob[k]) = lo[k];
        *reinterpret_cast<uint4*>(dst + ob[k] + 64) = hi[k];
      }
    }
    __syncthreads();  // this unit's rows are read; the next unit's are written
  }
  if (std::is_same<TOut, __half>::value && f16x2_has_inf(amax)) atomicOr(a.iws + FI_H_STATUS, kStatusRange);
}

inline int log2_of(int page_size) {
  int lp = 0;
  while ((1 << lp) < page_size) ++lp;
  return lp;
}

// Three CTAs per planned CTA of the run (the kernel's residency bound).
inline cudaError_t launch_rope_pass(const RopePass& rp, fi_dtype dtype, bool to_f16, int num_ctas, cudaStream_t s) {
  const unsigned grid = unsigned(3 * (num_ctas > 0 ? num_ctas : 1));
  if (dtype == FI_BF16 && to_f16)
    rope_pass_kernel<__nv_bfloat16, __half><<<grid, kRopeThreads, 0, s>>>(rp);
  else if (dtype == FI_BF16)
    rope_pass_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kRopeThreads, 0, s>>>(rp);
  else
    rope_pass_kernel<__half, __half><<<grid, kRopeThreads, 0, s>>>(rp);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_variant(const RunParams& p, int num_ctas, int variant, cudaStream_t s) {
  switch (variant & 7) {
    case 0: return launch_run<T, false, false, false>(p, num_ctas, s);
    case 1: return launch_run<T, true, false, false>(p, num_ctas, s);
    case 2: return launch_run<T, false, true, false>(p, num_ctas, s);
    case 3: return launch_run<T, true, true, false>(p, num_ctas, s);
    case 4: return launch_run<T, false, false, true>(p, num_ctas, s);
    case 5: return launch_run<T, true, false, true>(p, num_ctas, s);
    case 6: return launch_run<T, false, true, true>(p, num_ctas, s);
    default: return launch_run<T, true, true, true>(p, num_ctas, s);
  }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool stride_ok(int64_t elems) { return elems > 0 && (elems * 2) % 16 == 0; }

// cuTensorMapEncodeTiled, fetched through the runtime so the library does
// not link the driver library directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return EncodeTiledFn(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 16-bit tensor map; dims/strides innermost first, strides in elements (the
// innermost stride is 1).  Out-of-bounds boxes fill with zeros.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank, const uint64_t* dims,
              const int64_t* strides_elems, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = cuuint64_t(strides_elems[i]) * 2;
  return enc(map, type, cuuint32_t(rank), const_cast<void*>(base), gdim, gstride, bdim, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fi

using namespace fi;

extern "C" fi_status fi_default_plan_config(int device, fi_plan_config* out) {
  if (!out) return FI_ERR_INVALID_ARG;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return FI_ERR_CUDA;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return FI_ERR_CUDA;
  int per_sm = 0;
  const cudaError_t e = run_kernel_occupancy(&per_sm);
  cudaSetDevice(prev);
  if (e != cudaSuccess || per_sm < 1) return FI_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  out->num_ctas = sms * per_sm;
  out->max_batch = 8192;
  out->max_items = 1 << 17;
  out->max_merge_units = 1 << 15;
  out->max_partial_rows = int64_t(1) << 19;
  out->decode_min_chunk = 256;
  out->prefill_min_chunk = 1024;
  out->decode_cost_weight = 8;
  out->prefill_cost_weight = 9;
  out->split_factor = 1;
  out->window_left = -1;
  out->sink_tokens = 0;
  out->logits_soft_cap = 0.f;
  out->rope_max_positions = 0;
  out->rope_theta = 10000.f;
  out->rope_scale = 1.f;
  return FI_OK;
}

namespace fi {

// One KV cache given to a run: K and V [pages, P, Hkv, d] with their strides
// (elements) and the device page ids of the requests that read it.
struct CacheArgs {
  const void* k;
  const int64_t* k_strides;
  const void* v;
  const int64_t* v_strides;
  int32_t num_pages;
  const int32_t* kv_indices;
  int32_t page_size;
};

fi_status check_cache(const CacheArgs& c) {
  if (!c.k || !c.v || !c.k_strides || !c.v_strides || !c.kv_indices || c.num_pages < 1) return FI_ERR_INVALID_ARG;
  const int P = c.page_size;
  if (P < 1 || P > 128 || (P & (P - 1))) return FI_ERR_UNSUPPORTED;
  if (!aligned16(c.k) || !aligned16(c.v)) return FI_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (!stride_ok(c.k_strides[i]) || !stride_ok(c.v_strides[i])) return FI_ERR_ALIGNMENT;
  return FI_OK;
}

// The tensor maps of one cache.  Prefill-class items of a cache read it on
// the tensor cores when every TMA box of a page is a whole number of
// 1024-byte swizzle atoms (P >= 8) and a tile holds whole tokens (G divides
// 128); otherwise the CUDA-core path runs them.  K and V get maps of their
// own, each with its own strides: the copy engine does the page/slot/head
// address arithmetic for both, so equal and unequal K/V strides (the
// comparison of the BatchAttention PR page, "코드 분석 §2") take one path.
fi_status build_cache(KvCache* kc, const CacheArgs& c, CUtensorMapDataType tt, int32_t num_kv_heads, int32_t G) {
  const int P = c.page_size;
  kc->kv_indices = c.kv_indices;
  kc->page_size = P;
  int lp = 0;
  while ((1 << lp) < P) ++lp;
  kc->log2_page = lp;
  kc->num_pages = c.num_pages;
  kc->tc = (P >= kMinTmaPage && kTileM % G == 0) ? 1 : 0;
  const uint64_t kd[4] = {uint64_t(kHeadDim), uint64_t(num_kv_heads), uint64_t(P), uint64_t(c.num_pages)};
  const int64_t ks[3] = {c.k_strides[2], c.k_strides[1], c.k_strides[0]};  // head, slot, page
  const int64_t vs[3] = {c.v_strides[2], c.v_strides[1], c.v_strides[0]};
  const uint32_t kbd[4] = {uint32_t(kHeadDim), 1u, uint32_t(P < kStageTokens ? P : kStageTokens), 1u};
  if (!make_map(&kc->tm_kd, tt, c.k, 4, kd, ks, kbd, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&kc->tm_vd, tt, c.v, 4, kd, vs, kbd, CU_TENSOR_MAP_SWIZZLE_NONE))
    return FI_ERR_UNSUPPORTED;
  // Page size 1 where a page's stride is a whole number R >= Hkv of head
  // strides: each cache is a plain matrix of rows of 128 dims, row
  // page * R + head, and the decode stages fetch four rows per TMA gather
  // instead of one single-row box per token.
  auto rows_per_page = [&](const int64_t* st) -> int64_t {
    if (st[2] <= 0 || st[0] % st[2]) return 0;
    const int64_t r = st[0] / st[2];
    return (r >= num_kv_heads && (int64_t(c.num_pages) + 1) * r < (int64_t(1) << 31)) ? r : 0;
  };
  const int64_t rk = rows_per_page(c.k_strides), rv = rows_per_page(c.v_strides);
  if (P == 1 && rk > 0 && rv > 0) {
    const uint64_t gk[2] = {uint64_t(kHeadDim), uint64_t(c.num_pages) * uint64_t(rk)};
    const uint64_t gv[2] = {uint64_t(kHeadDim), uint64_t(c.num_pages) * uint64_t(rv)};
    const uint32_t gb[2] = {uint32_t(kHeadDim), 1u};
    if (!make_map(&kc->tm_kg, tt, c.k, 2, gk, &c.k_strides[2], gb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&kc->tm_vg, tt, c.v, 2, gv, &c.v_strides[2], gb, CU_TENSOR_MAP_SWIZZLE_NONE))
      return FI_ERR_UNSUPPORTED;
    kc->gather_rows = 1;
    kc->gather_rows_k = int32_t(rk);
    kc->gather_rows_v = int32_t(rv);
  }
  // Page size 1 with multi-head decode units (GQA groups a multiple of 4):
  // one box per token holds that token's rows of the unit's H KV heads.
  const int32_t mh = fi_mh_heads(G, num_kv_heads);
  if (P == 1 && mh > 1) {
    const uint32_t hb[4] = {uint32_t(kHeadDim), uint32_t(mh), 1u, 1u};
    if (!make_map(&kc->tm_kh, tt, c.k, 4, kd, ks, hb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&kc->tm_vh, tt, c.v, 4, kd, vs, hb, CU_TENSOR_MAP_SWIZZLE_NONE))
      return FI_ERR_UNSUPPORTED;
    kc->mh_heads = mh;
  }
  if (kc->tc) {
    const uint32_t kb[4] = {64u, 1u, uint32_t(P), 1u};
    if (!make_map(&kc->tm_k, tt, c.k, 4, kd, ks, kb, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&kc->tm_v, tt, c.v, 4, kd, vs, kb, CU_TENSOR_MAP_SWIZZLE_128B))
      return FI_ERR_UNSUPPORTED;
  }
  return FI_OK;
}

// Cascade merge (two-level plans), launched after the run on the same
// stream: for every entry and packed row, the LSE-weighted merge of the
// row's partial states -- its shared block's chunks, then its own request's
// chunks, in that order -- written as O and LSE.  One warp per (entry, row)
// task; an entry holds at most FI_CASCADE_ROWS rows, so the tasks are
// (entry, 0 .. FI_CASCADE_ROWS - 1) walked with a grid stride, and the counts
// come from the workspace header (a graph captured once replays correctly
// for any later cascade plan).  Lane l holds dims 4l..4l+3.  Nothing is
// written when the status word reports an error.
constexpr int kMergeGroup = 16;  // partial states whose O slices a merge lane loads at once

template <typename T>
__global__ void __launch_bounds__(256) cascade_merge_kernel(const int32_t* __restrict__ iws,
                                                            const float* __restrict__ fws, int64_t partial_o_offset,
                                                            T* o, int64_t o_stride_tok, int64_t o_stride_head,
                                                            float* lse, int num_qo_heads, int group) {
  const int lane = threadIdx.x & 31;
  // (entry, row) tasks, the plan's largest entry giving the row count of all.
  // The plan (copied in before the run) is read before the dependency wait,
  // the task's entry included; the status word and the partial rows, which
  // the run writes, after it.
  const int rows_max = iws[FI_H_CASCADE_ROWS_MAX];
  const int64_t tasks = int64_t(iws[FI_H_NUM_CASCADE]) * rows_max;
  const int32_t* ent = iws + iws[FI_H_OFF_CASCADE];
  const int32_t* reqs = iws + iws[FI_H_OFF_REQUESTS];
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  int64_t task = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int4 e0, e1, e2;  // {b, hk, row0, row1}, {n0, base0, stride0, n1}, {base1, stride1, 0, 0}
  int64_t qo_start = 0;
  auto load_entry = [&] {
    const int4* e4 = reinterpret_cast<const int4*>(ent + FI_CASCADE_INTS * (task / rows_max));
    e0 = __ldg(e4);
    e1 = __ldg(e4 + 1);
    e2 = __ldg(e4 + 2);
    qo_start = __ldg(reqs + FI_REQ_INTS * e0.x);
  };
  if (task < tasks) load_entry();
  grid_dependency_wait();  // launched early behind the run: its partial rows are written from here on
  if (iws[FI_H_STATUS] != 0) return;
  for (bool first = true; task < tasks; task += warps, first = false) {
    if (!first) load_entry();
    const int r = int(task % rows_max);
    if (r >= e0.w - e0.z) continue;
    const int n0 = e1.x, n = e1.x + e1.w;
    // part c (c < n): partial row of the row's c-th state
    auto part_row = [&](int c) -> int64_t {
      return c < n0 ? int64_t(e1.y) + int64_t(c) * e1.z + r : int64_t(e2.x) + int64_t(c - n0) * e2.y + r;
    };
    auto o_of = [&](int c) {
      return __ldcg(reinterpret_cast<const float4*>(fws + partial_o_offset + part_row(c) * kHeadDim) + lane);
    };
    // This lane's LSE (state `lane`) and the first kMergeGroup states' O
    // slices depend only on the entry: they go out together, so a row of at
    // most kMergeGroup states costs two dependent rounds (entry, states).
    const float lse_lane = lane < n ? __ldcg(fws + part_row(lane)) : -INFINITY;
    float4 v[kMergeGroup];
#pragma unroll
    for (int u = 0; u < kMergeGroup; ++u)
      if (u < n) v[u] = o_of(u);
    float M = lse_lane;
    for (int c0 = 32; c0 < n; c0 += 32)
      M = fmaxf(M, c0 + lane < n ? __ldcg(fws + part_row(c0 + lane)) : -INFINITY);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int c0 = 0; c0 < n; c0 += 32) {
        const float lse_c = c0 == 0 ? lse_lane : c0 + lane < n ? __ldcg(fws + part_row(c0 + lane)) : -INFINITY;
        const float w_mine = c0 + lane < n ? ex2((lse_c - M) * 1.4426950408889634f) : 0.f;
        const int cn = min(32, n - c0);
        for (int g0 = 0; g0 < cn; g0 += kMergeGroup) {
          if (c0 + g0 > 0) {  // later groups: their O slices now
#pragma unroll
            for (int u = 0; u < kMergeGroup; ++u)
              if (g0 + u < cn) v[u] = o_of(c0 + g0 + u);
          }
#pragma unroll
          for (int u = 0; u < kMergeGroup; ++u) {
            const float w = __shfl_sync(0xffffffffu, w_mine, (g0 + u) & 31);
            if (g0 + u < cn) {
              Ls += w;
              acc.x += w * v[u].x;
              acc.y += w * v[u].y;
              acc.z += w * v[u].z;
              acc.w += w * v[u].w;
            }
          }
        }
      }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    const int row = e0.z + r;
    const int t = row / group;
    const int head = e0.y * group + (row - t * group);
    const int64_t tok = qo_start + t;
    uint2 packed;
    packed.x = Elem<T>::from_float2(acc.x * inv, acc.y * inv);
    packed.y = Elem<T>::from_float2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(o + tok * o_stride_tok + int64_t(head) * o_stride_head + lane * 4) = packed;
    if (lane == 0 && lse) lse[tok * num_qo_heads + head] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
  }
}

template <typename T>
cudaError_t launch_cascade_merge(const RunParams& p, int32_t blocks, cudaStream_t s) {
  return launch_behind_run(cascade_merge_kernel<T>, blocks, 256, s, static_cast<const int32_t*>(p.iws),
                           static_cast<const float*>(p.fws), p.partial_o_offset, reinterpret_cast<T*>(p.o),
                           p.o_stride_tok, p.o_stride_head, p.lse, int(p.num_qo_heads), int(p.group));
}

// The run behind both entry points: the plan's own cache, and for a cascade
// plan the shared blocks' cache.
fi_status run_impl(const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                   int32_t q_num_tokens, const CacheArgs& own, const CacheArgs* shared, void* o,
                   int64_t o_stride_tok, int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale,
                   void* int_workspace_dev, void* float_workspace_dev, void* stream, void* k_rot = nullptr,
                   const int64_t* k_rot_strides = nullptr, void* q_rot = nullptr, int64_t q_rot_stride_tok = 0,
                   int64_t q_rot_stride_head = 0) {
  if (!info || !q || !o || !int_workspace_dev) return FI_ERR_INVALID_ARG;
  if (info->num_ctas < 1 || q_num_tokens < 1 || !std::isfinite(sm_scale)) return FI_ERR_INVALID_ARG;
  if (info->num_partial_rows > 0 && !float_workspace_dev) return FI_ERR_INVALID_ARG;
  if (info->num_shared > 0 && !shared) return FI_ERR_INVALID_ARG;  // a cascade plan needs the shared cache
  if (info->head_dim != kHeadDim) return FI_ERR_UNSUPPORTED;
  if (dtype != FI_FP16 && dtype != FI_BF16) return FI_ERR_UNSUPPORTED;
  if (info->num_kv_heads < 1 || info->num_qo_heads % info->num_kv_heads) return FI_ERR_UNSUPPORTED;
  fi_status st = check_cache(own);
  if (st == FI_OK && shared) st = check_cache(*shared);
  if (st != FI_OK) return st;
  if (!aligned16(q) || !aligned16(o) || !aligned16(int_workspace_dev) ||
      (float_workspace_dev && !aligned16(float_workspace_dev)) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FI_ERR_ALIGNMENT;
  if (!stride_ok(q_stride_tok) || !stride_ok(q_stride_head) || !stride_ok(o_stride_tok) || !stride_ok(o_stride_head))
    return FI_ERR_ALIGNMENT;

  RunParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const uint16_t*>(q);
  p.q_stride_tok = q_stride_tok;
  p.q_stride_head = q_stride_head;
  p.o = static_cast<uint16_t*>(o);
  p.o_stride_tok = o_stride_tok;
  p.o_stride_head = o_stride_head;
  p.lse = lse;
  p.iws = static_cast<int32_t*>(int_workspace_dev);
  p.fws = static_cast<float*>(float_workspace_dev);
  p.partial_o_offset = fi_partial_o_offset(info->max_partial_rows);
  p.max_partial_rows = p.fws ? info->max_partial_rows : 0;
  p.q_num_tokens = q_num_tokens;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.num_qo_heads = info->num_qo_heads;
  p.num_kv_heads = info->num_kv_heads;
  p.group = info->num_qo_heads / info->num_kv_heads;
  const int G = p.group;
  const CUtensorMapDataType tt = dtype == FI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  st = build_cache(&p.kv[0], own, tt, info->num_kv_heads, G);
  if (st == FI_OK && shared) {
    st = build_cache(&p.kv[1], *shared, tt, info->num_kv_heads, G);
    p.has_shared = 1;
  }
  if (st != FI_OK) return st;
  if (k_rot) {
    // RoPE with the queries and keys of prefill-class requests pre-rotated
    // into q_rot and k_rot (fp16): the tensor-core path reads them there; V,
    // and the CUDA-core path's queries and keys (rotated inside the kernel),
    // stay where they are.  A plan without prefill-class items (or pages
    // with no tensor-core path) makes this the fully fused run: no pass, and
    // a graph captured from it stays correct for any later plan (its
    // tensor-core items then rotate inside the kernel).
    if (!(info->variant & 4) || !k_rot_strides || !q_rot) return FI_ERR_INVALID_ARG;
    if (!aligned16(k_rot) || !aligned16(q_rot) || !stride_ok(q_rot_stride_tok) || !stride_ok(q_rot_stride_head))
      return FI_ERR_ALIGNMENT;
    for (int i = 0; i < 3; ++i)
      if (!stride_ok(k_rot_strides[i])) return FI_ERR_ALIGNMENT;
    if (p.kv[0].tc && info->num_prefill_items > 0) {
      const int P = own.page_size;
      const uint64_t kd[4] = {uint64_t(kHeadDim), uint64_t(info->num_kv_heads), uint64_t(P), uint64_t(own.num_pages)};
      const int64_t ks[3] = {k_rot_strides[2], k_rot_strides[1], k_rot_strides[0]};
      const uint32_t kb[4] = {64u, 1u, uint32_t(P), 1u};
      if (!make_map(&p.kv[0].tm_k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k_rot, 4, kd, ks, kb, CU_TENSOR_MAP_SWIZZLE_128B))
        return FI_ERR_UNSUPPORTED;
      p.qk_prerotated = 1;
    }
  }
  if (p.kv[0].tc || p.kv[1].tc) {
    const uint64_t qd[3] = {uint64_t(kHeadDim), uint64_t(info->num_qo_heads), uint64_t(q_num_tokens)};
    const int64_t qs[2] = {q_stride_head, q_stride_tok};
    const uint32_t qb[3] = {64u, uint32_t(G), uint32_t(kTileM / G)};
    const int64_t os[2] = {o_stride_head, o_stride_tok};
    const int64_t qrs[2] = {q_rot_stride_head, q_rot_stride_tok};
    const bool qr = p.qk_prerotated != 0;
    if (!make_map(&p.tm_q, qr ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : tt, qr ? q_rot : q, 3, qd, qr ? qrs : qs, qb,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_o, tt, o, 3, qd, os, qb, CU_TENSOR_MAP_SWIZZLE_128B))
      return FI_ERR_UNSUPPORTED;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The plan's variant picks the instantiation: bit 0 logits soft-cap, bit 1
  // sliding window / sink mask, bit 2 RoPE; the plain kernel carries none.
  // The late merge follows the run when the plan in `info` has late units;
  // a graph captured from a plan without any replays no late merge, and the
  // run then merges late units of later plans itself.  A cascade plan's
  // merge follows the run when `info` has cascade entries.
  p.late_merge = info->num_late_merge_units > 0 ? 1 : 0;
  cudaError_t e = cudaSuccess;
  int variant = info->variant;
  if (p.qk_prerotated) {
    RopePass rp{p.iws, static_cast<const uint16_t*>(own.k), {own.k_strides[0], own.k_strides[1], own.k_strides[2]},
                static_cast<uint16_t*>(k_rot), {k_rot_strides[0], k_rot_strides[1], k_rot_strides[2]},
                own.kv_indices, static_cast<const uint16_t*>(q), q_stride_tok, q_stride_head,
                static_cast<uint16_t*>(q_rot), q_rot_stride_tok, q_rot_stride_head, log2_of(own.page_size),
                info->num_kv_heads, info->num_qo_heads, G, 1, 1, 1};
    e = launch_rope_pass(rp, dtype, true, info->num_ctas, s);
    // With every item on the tensor-core path nothing is left to rotate in
    // the kernel: the instantiation without RoPE runs (it refuses a plan
    // with CUDA-core items, which a later re-plan could bring).
    if (info->num_decode_items == 0) variant &= ~4;
  }
  if (e == cudaSuccess)
    e = dtype == FI_BF16 ? launch_variant<__nv_bfloat16>(p, info->num_ctas, variant, s)
                         : launch_variant<__half>(p, info->num_ctas, variant, s);
  if (e == cudaSuccess && p.late_merge)
    e = dtype == FI_BF16 ? launch_late_merge<__nv_bfloat16>(p, 4 * info->num_ctas, s)
                         : launch_late_merge<__half>(p, 4 * info->num_ctas, s);
  if (e == cudaSuccess && info->num_cascade_merges > 0)
    e = dtype == FI_BF16 ? launch_cascade_merge<__nv_bfloat16>(p, 4 * info->num_ctas, s)
                         : launch_cascade_merge<__half>(p, 4 * info->num_ctas, s);
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

}  // namespace fi

extern "C" fi_status fi_batch_paged_attention_run(const fi_plan_info* info, const void* q, int64_t q_stride_tok,
                                                  int64_t q_stride_head, int32_t q_num_tokens, const void* k_cache,
                                                  const int64_t k_strides[3], const void* v_cache,
                                                  const int64_t v_strides[3], int32_t num_pages,
                                                  const int32_t* kv_indices_dev, void* o, int64_t o_stride_tok,
                                                  int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale,
                                                  void* int_workspace_dev, void* float_workspace_dev, void* stream) {
  if (!info) return FI_ERR_INVALID_ARG;
  const CacheArgs own{k_cache, k_strides, v_cache, v_strides, num_pages, kv_indices_dev, info->page_size};
  return run_impl(info, q, q_stride_tok, q_stride_head, q_num_tokens, own, nullptr, o, o_stride_tok, o_stride_head,
                  lse, dtype, sm_scale, int_workspace_dev, float_workspace_dev, stream);
}

extern "C" fi_status fi_batch_paged_attention_run_rope_prerotated(
    const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head, int32_t q_num_tokens,
    const void* k_cache, const int64_t k_strides[3], const void* v_cache, const int64_t v_strides[3],
    int32_t num_pages, const int32_t* kv_indices_dev, void* q_rot, int64_t q_rot_stride_tok,
    int64_t q_rot_stride_head, void* k_rot, const int64_t k_rot_strides[3], void* o, int64_t o_stride_tok,
    int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale, void* int_workspace_dev,
    void* float_workspace_dev, void* stream) {
  if (!info || !k_rot || !q_rot) return FI_ERR_INVALID_ARG;
  const CacheArgs own{k_cache, k_strides, v_cache, v_strides, num_pages, kv_indices_dev, info->page_size};
  return run_impl(info, q, q_stride_tok, q_stride_head, q_num_tokens, own, nullptr, o, o_stride_tok, o_stride_head,
                  lse, dtype, sm_scale, int_workspace_dev, float_workspace_dev, stream, k_rot, k_rot_strides, q_rot,
                  q_rot_stride_tok, q_rot_stride_head);
}

extern "C" fi_status fi_batch_paged_attention_run_cascade(
    const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head, int32_t q_num_tokens,
    const void* k_cache, const int64_t k_strides[3], const void* v_cache, const int64_t v_strides[3],
    int32_t num_pages, const int32_t* kv_indices_dev, const void* shared_k_cache, const int64_t shared_k_strides[3],
    const void* shared_v_cache, const int64_t shared_v_strides[3], int32_t shared_num_pages,
    const int32_t* shared_kv_indices_dev, int32_t shared_page_size, void* o, int64_t o_stride_tok,
    int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale, void* int_workspace_dev,
    void* float_workspace_dev, void* stream) {
  if (!info) return FI_ERR_INVALID_ARG;
  const CacheArgs own{k_cache, k_strides, v_cache, v_strides, num_pages, kv_indices_dev, info->page_size};
  const CacheArgs shared{shared_k_cache,   shared_k_strides, shared_v_cache,  shared_v_strides,
                         shared_num_pages, shared_kv_indices_dev, shared_page_size};
  return run_impl(info, q, q_stride_tok, q_stride_head, q_num_tokens, own, &shared, o, o_stride_tok, o_stride_head,
                  lse, dtype, sm_scale, int_workspace_dev, float_workspace_dev, stream);
}

extern "C" fi_status fi_rope_init(const fi_plan_config* cfg, void* int_workspace_dev, void* stream) {
  if (!cfg || !int_workspace_dev || cfg->rope_max_positions <= 0) return FI_ERR_INVALID_ARG;
  if (!(cfg->rope_theta > 0.f && cfg->rope_theta < HUGE_VALF && cfg->rope_scale > 0.f && cfg->rope_scale < HUGE_VALF))
    return FI_ERR_INVALID_ARG;
  if (!aligned16(int_workspace_dev)) return FI_ERR_ALIGNMENT;
  float2* table = reinterpret_cast<float2*>(static_cast<char*>(int_workspace_dev) +
                                            fi_rope_table_offset(plan_capacity_ints(cfg)));
  const int64_t entries = fi_rope_table_rows(cfg->rope_max_positions) * FI_ROPE_PAIRS;
  const int64_t blocks = (entries + 255) / 256;
  rope_table_kernel<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      table, entries, double(cfg->rope_theta), 1.0 / double(cfg->rope_scale));
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

extern "C" fi_status fi_rope_apply_k(const fi_plan_info* info, void* int_workspace_dev, const void* k_in,
                                     const int64_t k_in_strides[3], void* k_out, const int64_t k_out_strides[3],
                                     const int32_t* kv_indices_dev, fi_dtype dtype, void* stream) {
  if (!info || !int_workspace_dev || !k_in || !k_out || !k_in_strides || !k_out_strides || !kv_indices_dev)
    return FI_ERR_INVALID_ARG;
  if (!(info->variant & 4) || info->num_shared > 0) return FI_ERR_INVALID_ARG;  // no RoPE table, or two caches
  if (info->head_dim != kHeadDim) return FI_ERR_UNSUPPORTED;
  if (dtype != FI_FP16 && dtype != FI_BF16) return FI_ERR_UNSUPPORTED;
  if (!aligned16(k_in) || !aligned16(k_out) || !aligned16(int_workspace_dev)) return FI_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (!stride_ok(k_in_strides[i]) || !stride_ok(k_out_strides[i])) return FI_ERR_ALIGNMENT;
  if (info->batch == 0) return FI_OK;
  const RopePass rp{static_cast<int32_t*>(int_workspace_dev), static_cast<const uint16_t*>(k_in),
                    {k_in_strides[0], k_in_strides[1], k_in_strides[2]}, static_cast<uint16_t*>(k_out),
                    {k_out_strides[0], k_out_strides[1], k_out_strides[2]}, kv_indices_dev, nullptr, 0, 0, nullptr,
                    0, 0, log2_of(info->page_size), info->num_kv_heads, info->num_qo_heads,
                    info->num_qo_heads / info->num_kv_heads, 1, 0, 0};
  return launch_rope_pass(rp, dtype, false, info->num_ctas, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FI_OK
             : FI_ERR_CUDA;
}

extern "C" fi_status fi_rope_apply_q(const fi_plan_info* info, void* int_workspace_dev, const void* q_in,
                                     int64_t q_in_stride_tok, int64_t q_in_stride_head, void* q_out,
                                     int64_t q_out_stride_tok, int64_t q_out_stride_head, fi_dtype dtype,
                                     void* stream) {
  if (!info || !int_workspace_dev || !q_in || !q_out) return FI_ERR_INVALID_ARG;
  if (!(info->variant & 4) || info->num_shared > 0) return FI_ERR_INVALID_ARG;
  if (info->head_dim != kHeadDim) return FI_ERR_UNSUPPORTED;
  if (dtype != FI_FP16 && dtype != FI_BF16) return FI_ERR_UNSUPPORTED;
  if (!aligned16(q_in) || !aligned16(q_out) || !aligned16(int_workspace_dev)) return FI_ERR_ALIGNMENT;
  if (!stride_ok(q_in_stride_tok) || !stride_ok(q_in_stride_head) || !stride_ok(q_out_stride_tok) ||
      !stride_ok(q_out_stride_head))
    return FI_ERR_ALIGNMENT;
  if (info->batch == 0) return FI_OK;
  const RopePass rp{static_cast<int32_t*>(int_workspace_dev), nullptr, {0, 0, 0}, nullptr, {0, 0, 0}, nullptr,
                    static_cast<const uint16_t*>(q_in), q_in_stride_tok, q_in_stride_head,
                    static_cast<uint16_t*>(q_out), q_out_stride_tok, q_out_stride_head, log2_of(info->page_size),
                    info->num_kv_heads, info->num_qo_heads, info->num_qo_heads / info->num_kv_heads, 0, 1, 0};
  return launch_rope_pass(rp, dtype, false, info->num_ctas, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FI_OK
             : FI_ERR_CUDA;
}

extern "C" fi_status fi_merge_states(const void* v_a, const float* s_a, const void* v_b, const float* s_b,
                                     void* v_out, float* s_out, int32_t rows, int32_t heads, int32_t head_dim,
                                     fi_dtype dtype, void* stream) {
  if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out || rows < 0 || heads < 1) return FI_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return FI_ERR_UNSUPPORTED;
  if (dtype != FI_FP16 && dtype != FI_BF16 && dtype != FI_FP32) return FI_ERR_UNSUPPORTED;
  if (!aligned16(v_a) || !aligned16(v_b) || !aligned16(v_out)) return FI_ERR_ALIGNMENT;
  const int64_t states = int64_t(rows) * heads;
  if (states == 0) return FI_OK;
  const int64_t blocks = (states * 16 + 255) / 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case FI_BF16:
      merge_states_kernel<__nv_bfloat16><<<unsigned(blocks), 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(v_a), s_a, static_cast<const __nv_bfloat16*>(v_b), s_b,
          static_cast<__nv_bfloat16*>(v_out), s_out, states);
      break;
    case FI_FP16:
      merge_states_kernel<__half><<<unsigned(blocks), 256, 0, s>>>(static_cast<const __half*>(v_a), s_a,
                                                                   static_cast<const __half*>(v_b), s_b,
                                                                   static_cast<__half*>(v_out), s_out, states);
      break;
    default:
      merge_states_kernel<float><<<unsigned(blocks), 256, 0, s>>>(static_cast<const float*>(v_a), s_a,
                                                                  static_cast<const float*>(v_b), s_b,
                                                                  static_cast<float*>(v_out), s_out, states);
  }
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

namespace fi {

// One warp waits, through the same bounded wait the kernels use, on an
// mbarrier nothing arrives on: the wait gives up after its budget, and the
// status word records the timeout exactly as a stalled kernel role would.
__global__ void bounded_wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = warp_wait(&bar, 0, &abort_flag);
  if (threadIdx.x == 0 && !ok) atomicOr(status, abort_flag);
}

}  // namespace fi

extern "C" fi_status fi_selftest_bounded_wait(void* int_workspace_dev, void* stream) {
  if (!int_workspace_dev) return FI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(int_workspace_dev) & 15u) return FI_ERR_ALIGNMENT;
  fi::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(int_workspace_dev) + FI_H_STATUS);
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

extern "C" fi_status fi_get_device_status(const void* int_workspace_dev, void* stream, int32_t* status_out) {
  if (!int_workspace_dev || !status_out) return FI_ERR_INVALID_ARG;
  int32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, static_cast<const int32_t*>(int_workspace_dev) + FI_H_STATUS, sizeof word,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FI_ERR_CUDA;
  *status_out = (word & kStatusTimeout)                   ? FI_ERR_TIMEOUT
                : (word & (kStatusBadPlan | kStatusRange)) ? FI_ERR_DEVICE_CHECK
                                                           : FI_OK;
  return FI_OK;
}

// ------------------------------------------------------------ run without caller scratch

// Some callers cannot hand the library a float workspace: code that runs
// where no device allocator is reachable (a plugin given fixed input/output
// buffers by its host runtime, a server that reserved all device memory up
// front and owns no spare block), or code that must not allocate at that
// point because an allocation would synchronise the device or be recorded
// into a stream it does not control.  For them the split-KV partial states
// live in one fixed device array defined here, sized for at most
// kStaticPartialRows partial rows (about 17 MB, held by every GPU that loads
// this library until the process exits).
namespace fi {
constexpr int64_t kStaticPartialRows = 32768;  // a multiple of 64: partial O starts right after the LSEs
constexpr int64_t kStaticScratchFloats = kStaticPartialRows + kStaticPartialRows * kHeadDim;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

std::mutex g_static_scratch_mu;
float* g_static_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up once
// per device (in host code the symbol is only a stand-in, not an address).
fi_status static_scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FI_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return FI_ERR_CUDA;
    g_static_scratch_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_static_scratch_ptr[dev];
  return FI_OK;
}
}  // namespace fi

extern "C" fi_status fi_batch_paged_attention_run_static_scratch(
    const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head, int32_t q_num_tokens,
    const void* k_cache, const int64_t k_strides[3], const void* v_cache, const int64_t v_strides[3],
    int32_t num_pages, const int32_t* kv_indices_dev, void* o, int64_t o_stride_tok, int64_t o_stride_head,
    float* lse, fi_dtype dtype, float sm_scale, void* int_workspace_dev, void* stream) {
  if (!info) return FI_ERR_INVALID_ARG;
  if (info->num_partial_rows > kStaticPartialRows) return FI_ERR_CAPACITY;  // plan needs more partial rows
  float* scratch = nullptr;
  const fi_status st = static_scratch_address(&scratch);
  if (st != FI_OK) return st;
  // The same run as fi_batch_paged_attention_run, with the fixed array as
  // its float workspace (laid out for kStaticPartialRows rows).  Nothing in
  // that array has to start at zero: every partial row is written before it
  // is read, and the merge counters live in the caller's int workspace.
  fi_plan_info local = *info;
  local.max_partial_rows = kStaticPartialRows;
  return fi_batch_paged_attention_run(&local, q, q_stride_tok, q_stride_head, q_num_tokens, k_cache, k_strides,
                                      v_cache, v_strides, num_pages, kv_indices_dev, o, o_stride_tok, o_stride_head,
                                      lse, dtype, sm_scale, int_workspace_dev, scratch, stream);
}
