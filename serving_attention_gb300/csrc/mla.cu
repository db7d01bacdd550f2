// mla.cu -- absorbed-MLA decode on the 5th-generation tensor cores.
//
// FlashInfer 0.6 wiki page, section "MLA(Multi-head Latent Attention) 커널":
// the cache holds one 512-dim latent per token (plus a 64-dim RoPE key shared
// by the heads) and the up-projections are folded into the attention, so the
// kernel attends over the latents directly:
//   s_hj = scale * (q_nope_h . c_j + q_pe_h . r_j),   o_h = sum_j p_hj c_j.
// The same wiki page, section "Blackwell (SM100/SM103) 전용 경로 / SM103
// (B300) MLA 디코드", describes the B300 path as a cluster-aware split-KV
// decode.  This kernel's own design for sm_103a:
//
//  * one tile = the 128 query heads of one request (the MMA's M = 128;
//    fewer heads are zero rows) against 64-token KV blocks;
//  * a thread-block cluster of two CTAs per KV chunk.  The fp32 output tile
//    of 128 heads x 512 dims would fill all 512 TMEM columns of one SM and
//    leave none for the logits, so CTA r of the pair owns output dims
//    [256 r, 256 r + 256) (256 columns) and double-buffers the logits S in
//    two 64-column buffers;
//  * the QK contraction is split the same way: CTA r multiplies latent dims
//    [256 r, 256 r + 256) and RoPE dims [32 r, 32 r + 32), so every byte of
//    the cache is read by exactly one CTA of the pair.  Each CTA sends its
//    64 partial logits per row to the other through distributed shared
//    memory and adds the other's: both then hold the same full S (fp32
//    addition is commutative, so bit for bit the same), take the same
//    softmax decisions, and accumulate P V into their own half of O;
//  * tensor memory holds O (256 columns), the two S buffers (64 each) and the
//    CTA's latent half of Q (256 bf16 dims per row, 128 columns), so shared
//    memory keeps only the RoPE quarter of Q, four KV stages and two 32 KB
//    exchange buffers;
//  * roles per CTA: warp 0 loads the RoPE part of Q and the KV blocks with TMA;
//    warp 1 issues the MMAs (S = Q K^T over 288 dims into TMEM, the latent part
//    with Q read from TMEM, then O += P V with P read from TMEM over the S
//    columns, N = 256); warps 4..7 write Q into TMEM, run the softmax (one head
//    row per thread = one TMEM lane) and the epilogue; warps 8..11 send each
//    block's partial logits to the partner as soon as S is in TMEM;
//  * S runs one block ahead of the softmax (S of block j + 2 is issued right
//    after P V of block j, into the buffer P of block j occupied), so the
//    softmax of one block overlaps the MMAs of the next; the rare lazy
//    rescale of O waits for the P V in flight first;
//  * a request cut into several chunks writes fp32 partial states that
//    mla_merge_kernel combines (LSE-weighted).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/fi_mla.h"
#include "mla_layout.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace fi {

// 16-bit tensor map (attention.cu): dims and strides innermost first, strides
// in elements; out-of-bounds boxes fill with zeros.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank, const uint64_t* dims,
              const int64_t* strides_elems, const uint32_t* box, CUtensorMapSwizzle swizzle);

namespace mla {

constexpr int kRows = FI_MLA_ROWS;          // heads per tile (MMA M)
constexpr int kDc = FI_MLA_LATENT_DIM;      // 512
constexpr int kHalf = kDc / 2;              // latent dims per CTA of the pair
constexpr int kRopeHalf = FI_MLA_ROPE_DIM / 2;  // RoPE dims per CTA
constexpr int kBlk = FI_MLA_BLOCK;          // KV tokens per block
constexpr int kGroups = kHalf / 64;         // 128-byte swizzled column groups of a CTA's latent half
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kAllocWarp = 2, kSoftmaxWarp0 = 4, kExchangeWarp0 = 8;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;  // O: 0..255; S buffers: 256..319, 320..383; Q: 384..511
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemQ = 384;
constexpr float kLazyRescale = 8.0f;  // log2 units: keep a stale max until it is 2^8 off
constexpr int kMergeThreads = 128;
constexpr int kMergeBlocksPerPair = 32;

// One KV block of this CTA's half: the latent rows as 4 groups of 64 dims
// (128-byte rows, 128-byte swizzle, 8 KB each) and the RoPE rows (64-byte
// rows, 64-byte swizzle).  Row t = token t of the block.
struct Stage {
  uint16_t lat[kGroups][kBlk][64];
  uint16_t rope[kBlk][kRopeHalf];
};

struct Smem {
  uint16_t q_rope[kRows][kRopeHalf];   // this CTA's RoPE quarter of the 128 query rows
  Stage st[kStages];
  uint4 xbuf[2][kBlk / 4][kRows];      // the partner's partial logits of block g in buffer g % 2: chunk
                                       // q (logits 4q..4q+3) of row r at [q][r], so a warp's stores are
                                       // 512 contiguous bytes
  uint64_t full[kStages], empty[kStages];
  uint64_t q_full;                     // the RoPE part of Q has landed (TMA)
  uint64_t q_lat_full;                 // the latent part of Q is in TMEM (the 4 softmax warps)
  uint64_t q_empty;                    // the chunk's last S has completed (MMA commit)
  uint64_t s_full[2];                  // S buffer b holds the logits of a block (MMA commit)
  uint64_t p_full;                     // P of the current block is in TMEM (the 4 softmax warps)
  uint64_t pv_done;                    // P V of a block has completed (MMA commit)
  uint64_t o_ready, o_free;            // O of a chunk complete / read out by the epilogue
  uint64_t xfull[2];                   // the partner's logits have landed in xbuf[b] (32 KB of complete_tx)
  uint64_t xfree[2];                   // the partner's 4 softmax warps read the logits sent into their xbuf[b]
  uint64_t s_read[2];                  // the exchange warps have read S buffer b (P may overwrite it)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
static_assert(offsetof(Smem, q_rope) % 1024 == 0 && offsetof(Smem, st) % 1024 == 0 && sizeof(Stage) % 1024 == 0 &&
                  offsetof(Stage, rope) % 1024 == 0,
              "swizzled operand blocks start on 1024-byte boundaries");
constexpr uint32_t kQBytes = kRows * kRopeHalf * 2;  // one load of the RoPE part of Q
constexpr uint32_t kRowBytes = kGroups * 128 + kRopeHalf * 2;                // one token of a KV block

struct Params {
  CUtensorMap tm_qp;   // q_pe   [rows][heads][64],  box 32 x 128 x 1, 64-byte swizzle
  CUtensorMap tm_ckv;  // ckv    [pages][P][512],    box 64 x P x 1, 128-byte swizzle
  CUtensorMap tm_kpe;  // kpe    [pages][P][64],     box 32 x P x 1, 64-byte swizzle
  const uint16_t* q_nope;  // [rows][heads][512] bf16, element strides below
  int64_t qn_stride_tok, qn_stride_head;
  const int32_t* iws;
  int32_t* status;
  const int32_t* kv_indices;
  float* fws;
  int64_t partial_o_offset;
  int64_t max_parts;   // partial-state slots the float workspace holds
  int32_t q_rows;      // rows of the queries and outputs
  uint16_t* o;         // [rows][heads][512] bf16
  float* lse;          // [rows][heads] or null
  float scale_log2;
  int32_t num_heads;
  int32_t page_size;
};

// ---------------------------------------------------------------- cluster PTX

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Asynchronous store into another CTA's shared memory that, once it has
// landed, completes its 16 bytes on that CTA's barrier `remote_bar` (no fence
// in the issuing thread: the receiver's wait on the barrier orders the data).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(remote_bar)
               : "memory");
}

// Arrive on a barrier of another CTA of the cluster without a fence.  Used
// only to say "this warp has read its buffer", after an instruction that
// consumed every loaded value has issued: those loads have returned, so no
// later write of the other CTA can change what they read.  A release arrive
// would order the same thing at the cost of a cluster-scope fence (measured:
// about 2,300 SM cycles per block on the critical path).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded warp-wide wait on a phase completed by the other CTA's threads:
// every lane must see the completion itself (its own acquire), so the data
// the other CTA released is visible to each lane that reads it.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (__all_sync(0xffffffffu, mbar_try_wait_acq_cluster(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < kPollsPerCheck; ++k)
      if (__all_sync(0xffffffffu, mbar_try_wait_acq_cluster(bar, parity))) return true;
    const int gave_up = *abort != 0 ? 2 : 0;
    const int late = clock64() - t0 > kWaitBudgetClocks ? 4 : 0;
    const int st = __shfl_sync(0xffffffffu, gave_up | late, 0);
    if (st & 2) return false;
    if (st & 4) {
      *abort = kStatusTimeout;
      return false;
    }
  }
}

// Both CTAs of the cluster reach this point (all threads) before either goes on.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory descriptor of a K-major operand with 64-byte swizzle (rows of
// 64 bytes, 8-row groups 512 bytes apart): the layout field is 4.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t sbo_bytes) {
  return uint64_t((saddr >> 4) & 0x3FFF) | (uint64_t(1) << 16) | (uint64_t((sbo_bytes >> 4) & 0x3FFF) << 32) |
         (uint64_t(1) << 46) | (uint64_t(4) << 61);
}

struct Unit {
  int32_t b, kv0, kv1, part;
};

__device__ __forceinline__ Unit load_unit(const int32_t* iws, int32_t off_units, int32_t i) {
  const int4 v = __ldg(reinterpret_cast<const int4*>(iws + off_units) + i);
  return Unit{v.x, v.y, v.z, v.w};
}

__device__ __forceinline__ int unit_blocks(const Unit& u) { return (u.kv1 - u.kv0 + kBlk - 1) / kBlk; }

// ---------------------------------------------------------------- roles

// Warp 0: Q of each chunk, then its KV blocks through the stage ring.  Lane i
// loads page i of a block (a block holds 64 / page_size pages).
__device__ void producer(const Params& p, Smem& sm, uint32_t rank, int32_t begin, int32_t end, int32_t off_units,
                         int32_t off_req) {
  const int lane = threadIdx.x & 31;
  const int P = p.page_size;
  const int x_lat = kHalf * int(rank), x_rope = kRopeHalf * int(rank);
  int it = 0, nu = 0;
  int armed[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) armed[s] = -1;
  int q_armed = -1;
  bool ok = true;
  for (int32_t i = begin; i < end && ok; ++i) {
    const Unit u = load_unit(p.iws, off_units, i);
    const int32_t page_start = __ldg(p.iws + off_req + FI_MLA_REQ_INTS * u.b);
    ok = warp_wait(&sm.q_empty, (nu & 1) ^ 1, &sm.abort);
    if (!ok) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sm.q_full, kQBytes);
      tc::tma_load_3d(&sm.q_rope[0][0], &p.tm_qp, &sm.q_full, x_rope, 0, u.b);
    }
    q_armed = nu & 1;
    ++nu;
    const int nb = unit_blocks(u);
    for (int j = 0; j < nb; ++j, ++it) {
      const int s = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      ok = warp_wait(&sm.empty[s], ph ^ 1, &sm.abort);
      if (!ok) break;
      const int t0 = u.kv0 + j * kBlk;
      const int t1 = min(u.kv1, t0 + kBlk);
      const int npg = (t1 - t0 + P - 1) / P;  // t0 is a multiple of 64, hence of P
      if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], uint32_t(npg * P) * kRowBytes);
      __syncwarp();
      if (lane < npg) {
        const int32_t page = __ldg(p.kv_indices + page_start + t0 / P + lane);
        const int row = lane * P;
#pragma unroll
        for (int a = 0; a < kGroups; ++a)
          tc::tma_load_3d(&sm.st[s].lat[a][row][0], &p.tm_ckv, &sm.full[s], x_lat + 64 * a, 0, page);
        tc::tma_load_3d(&sm.st[s].rope[row][0], &p.tm_kpe, &sm.full[s], x_rope, 0, page);
      }
      armed[s] = int(ph);
    }
  }
  // every load this warp armed has landed before the CTA leaves
  if (lane == 0) {
    if (q_armed >= 0) mbar_wait_drain(&sm.q_full, uint32_t(q_armed));
    for (int s = 0; s < kStages; ++s)
      if (armed[s] >= 0) mbar_wait_drain(&sm.full[s], uint32_t(armed[s]));
  }
  __syncwarp();
}

// Warp 1: the MMAs.  Per chunk: S of blocks 0 and 1, then for each block j
// P V of block j followed by S of block j + 2 (same S buffer: the tensor pipe
// reads P of block j before it overwrites the buffer).
__device__ void mma_issuer(const Params& p, Smem& sm, int32_t begin, int32_t end, int32_t off_units) {
  const int lane = threadIdx.x & 31;
  constexpr uint32_t idesc_s = tc::idesc_f16(true, false, kRows, kBlk);
  constexpr uint32_t idesc_pv = tc::idesc_f16(true, true, kRows, kHalf);
  const uint32_t tmem = sm.tmem_base;
  // Descriptors of the first block of each operand; the start-address field
  // counts 16-byte units: a KV column group is 8 KB (512), a stage
  // sizeof(Stage) / 16, 16 dims along a swizzled row 32 bytes (2), 16 V tokens
  // 2 KB (128).  The latent part of Q is the A operand in TMEM: 16 dims are 8
  // columns of 16-bit pairs.  Every sum is a real shared-memory
  // address below 2^18 bytes, so the field never carries.
  const uint64_t dqr = smem_desc_sw64(smem_u32(&sm.q_rope[0][0]), 512);
  const uint64_t dk = tc::smem_desc_sw128(smem_u32(&sm.st[0].lat[0][0][0]), 16, 1024);
  const uint64_t dkr = smem_desc_sw64(smem_u32(&sm.st[0].rope[0][0]), 512);
  // V = the latent rows as an MN-major B operand: the next 64 dims 8 KB on
  const uint64_t dv = tc::smem_desc_sw128(smem_u32(&sm.st[0].lat[0][0][0]), kBlk * 128, 1024);
  constexpr uint32_t kStageUnits = uint32_t(sizeof(Stage) >> 4);
  bool issued = false, ok = true;
  int g = 0, nu = 0;  // blocks and chunks so far

  // waits for KV block gb and clears the rows past the chunk's end, so that
  // P = 0 never meets a non-finite value there in P V
  auto wait_block = [&](int gb, int ntok) -> bool {
    const int s = gb % kStages;
    if (!warp_wait(&sm.full[s], (gb / kStages) & 1, &sm.abort)) return false;
    if (ntok < kBlk) {
      uint4* base = reinterpret_cast<uint4*>(&sm.st[s].lat[0][0][0]);
      const int rows = kBlk - ntok;
      for (int e = lane; e < kGroups * rows * 8; e += 32) {
        const int a = e / (rows * 8), rem = e - a * rows * 8;
        base[(a * kBlk + ntok + rem / 8) * 8 + (rem & 7)] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    tc::fence_after_sync();
    return true;
  };
  auto issue_s = [&](int gb) {
    const uint32_t s = uint32_t(gb % kStages);
    const uint32_t d = tmem + kTmemS + 64u * uint32_t(gb & 1);
    const uint64_t k0 = dk + kStageUnits * s, r0 = dkr + kStageUnits * s;
#pragma unroll
    for (int kk = 0; kk < kHalf / 16; ++kk) {
      const uint32_t sk = 512u * uint32_t(kk >> 2) + 2u * uint32_t(kk & 3);
      tc::mma_ts_warp(d, tmem + kTmemQ + 8u * kk, k0 + sk, idesc_s, kk > 0 ? 1u : 0u);
    }
#pragma unroll
    for (int kk = 0; kk < kRopeHalf / 16; ++kk) tc::mma_ss_warp(d, dqr + 2u * kk, r0 + 2u * kk, idesc_s, 1u);
    tc::mma_commit_warp(&sm.s_full[gb & 1]);
    issued = true;
  };

  for (int32_t i = begin; i < end && ok; ++i) {
    const Unit u = load_unit(p.iws, off_units, i);
    const int nb = unit_blocks(u);
    auto ntok = [&](int j) { return min(kBlk, u.kv1 - (u.kv0 + j * kBlk)); };
    ok = warp_wait_all(2, &sm.q_full, nu & 1, &sm.q_lat_full, nu & 1, nullptr, 0, nullptr, 0, &sm.abort);
    if (!ok) break;
    tc::fence_after_sync();
    for (int j = 0; j < nb && j < 2 && ok; ++j) {
      ok = wait_block(g + j, ntok(j));
      if (!ok) break;
      issue_s(g + j);
      if (j == nb - 1) tc::mma_commit_warp(&sm.q_empty);  // the chunk's last read of Q
    }
    for (int j = 0; j < nb && ok; ++j) {
      const int gb = g + j;
      ok = warp_wait(&sm.p_full, gb & 1, &sm.abort);
      if (ok && j == 0) ok = warp_wait(&sm.o_free, (nu & 1) ^ 1, &sm.abort);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t s = uint32_t(gb % kStages);
      const uint32_t pcol = tmem + kTmemS + 64u * uint32_t(gb & 1);
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)  // P of tokens 16kk..16kk+15: 16-bit pairs in columns 8kk..8kk+7
        tc::mma_ts_warp(tmem, pcol + 8u * kk, dv + kStageUnits * s + 128u * kk, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit_warp(&sm.pv_done);
      tc::mma_commit_warp(&sm.empty[s]);
      if (j + 2 < nb) {
        ok = wait_block(gb + 2, ntok(j + 2));
        if (!ok) break;
        issue_s(gb + 2);
        if (j + 2 == nb - 1) tc::mma_commit_warp(&sm.q_empty);
      }
    }
    if (!ok) break;
    tc::mma_commit_warp(&sm.o_ready);
    g += nb;
    ++nu;
  }
  // no MMA may still run when the CTA frees its tensor memory
  if (issued) {
    tc::mma_commit_warp(&sm.drain);
    if (lane == 0) mbar_wait_drain(&sm.drain, 0);
    __syncwarp();
  }
}

// Warps 4..7: thread r owns head row r (TMEM lane r).  Per block: read this
// CTA's partial logits, send them to the partner, add the partner's, then the
// online softmax (log2 domain, lazy rescale) and P into TMEM; per chunk the
// epilogue of this CTA's 256 output dims.
__device__ void softmax_role(const Params& p, Smem& sm, uint32_t rank, int32_t begin, int32_t end,
                             int32_t off_units) {
  const int w = (threadIdx.x >> 5) - kSoftmaxWarp0;  // == warp % 4: TMEM lanes 32w..32w+31
  const int lane = threadIdx.x & 31;
  const int r = 32 * w + lane;
  const uint32_t tl = sm.tmem_base + (uint32_t(32 * w) << 16);
  const float c = p.scale_log2;
  const uint32_t peer = rank ^ 1u;
  const uint32_t xfree_remote[2] = {mapa_shared(smem_u32(&sm.xfree[0]), peer),
                                    mapa_shared(smem_u32(&sm.xfree[1]), peer)};
  const bool row_ok = r < p.num_heads;
  int g = 0, nu = 0;
  bool ok = true;
  for (int32_t i = begin; i < end && ok; ++i) {
    const Unit u = load_unit(p.iws, off_units, i);
    const int nb = unit_blocks(u);
    // The chunk's query rows into TMEM once the previous chunk's last S has
    // read them: this CTA's 256 latent dims of row r as 128 columns of pairs
    // (rows past the heads are zeros).
    ok = warp_wait(&sm.q_empty, (nu & 1) ^ 1, &sm.abort);
    if (!ok) break;
    // q_empty completes through the MMA warp's tcgen05.commit; the fence
    // orders this warp's tensor-memory stores below after that wait, so no
    // store can overtake an S MMA of the previous chunk still reading Q.
    tc::fence_after_sync();
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q_nope + int64_t(u.b) * p.qn_stride_tok +
                                                        int64_t(row_ok ? r : 0) * p.qn_stride_head) +
                         kHalf / 8 * int(rank);
      uint32_t qv[4][32];
#pragma unroll
      for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = row_ok ? __ldg(src + 8 * h + e) : make_uint4(0u, 0u, 0u, 0u);
          qv[h][4 * e] = v.x;
          qv[h][4 * e + 1] = v.y;
          qv[h][4 * e + 2] = v.z;
          qv[h][4 * e + 3] = v.w;
        }
#pragma unroll
      for (int h = 0; h < 4; ++h) tc::tmem_st32(tl + kTmemQ + 32u * h, qv[h]);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_lat_full);
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nb; ++j) {
      const int gb = g + j;
      const uint32_t scol = tl + kTmemS + 64u * uint32_t(gb & 1);
      ok = warp_wait(&sm.s_full[gb & 1], (gb >> 1) & 1, &sm.abort);
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t sv[2][32];
      tc::tmem_ld32(scol, sv[0]);
      tc::tmem_ld32(scol + 32, sv[1]);
      tc::tmem_ld_wait();
      // the partner's half of the logits, sent by its exchange warps
      const int xb = gb & 1;
      ok = warp_wait_cluster(&sm.xfull[xb], (gb >> 1) & 1, &sm.abort);
      if (!ok) break;
      float s[kBlk];
#pragma unroll
      for (int q = 0; q < kBlk / 4; ++q) {
        const uint4 x = sm.xbuf[xb][q][r];
        const uint32_t* v = &sv[q >> 3][4 * (q & 7)];
        s[4 * q + 0] = __uint_as_float(v[0]) + __uint_as_float(x.x);
        s[4 * q + 1] = __uint_as_float(v[1]) + __uint_as_float(x.y);
        s[4 * q + 2] = __uint_as_float(v[2]) + __uint_as_float(x.z);
        s[4 * q + 3] = __uint_as_float(v[3]) + __uint_as_float(x.w);
      }
      // Arm the buffer's next use (block gb + 2): its phase for block gb has
      // completed, and the partner sends block gb + 2 only after this warp's
      // signal below.
      if (r == 0) mbar_arrive_expect_tx(&sm.xfull[xb], kRows * kBlk * 4);
      const int ntok = min(kBlk, u.kv1 - (u.kv0 + j * kBlk));
      if (ntok < kBlk) {
#pragma unroll
        for (int e = 0; e < kBlk; ++e)
          if (e >= ntok) s[e] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx8[a] = s[a];
#pragma unroll
      for (int e = 8; e < kBlk; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], s[e]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * c;
      const float m_new = (mx > m + kLazyRescale) ? mx : m;
      const bool rescale = (m_new != m) && j > 0;
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds P V of the chunk's earlier blocks; the last of them may
        // still run (S of this block was issued after P V of block gb - 2)
        ok = warp_wait(&sm.pv_done, (gb - 1) & 1, &sm.abort);
        if (!ok) break;
        tc::fence_after_sync();
        const float alpha = rescale ? ex2(m - m_new) : 1.f;
#pragma unroll 1
        for (int h = 0; h < kHalf / 32; ++h) {
          uint32_t ov[32];
          tc::tmem_ld32(tl + 32u * h, ov);
          tc::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tc::tmem_st32(tl + 32u * h, ov);
        }
        tc::tmem_st_wait();
        if (rescale) l *= alpha;
      }
      const float msub = (m_new == -INFINITY) ? 0.f : m_new;
      const float2 cc = make_float2(c, c), nms = make_float2(-msub, -msub);
      float2 sum4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sum4[a] = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float2 x = fma2(make_float2(s[2 * e], s[2 * e + 1]), cc, nms);
        const float2 pe = make_float2(ex2(x.x), ex2(x.y));
        sum4[e & 3] = add2(sum4[e & 3], pe);
        pk[e] = tc::pack2<__nv_bfloat16>(pe.x, pe.y);
      }
      // P overwrites the S buffer once this CTA's exchange warps have read it
      ok = warp_wait(&sm.s_read[gb & 1], (gb >> 1) & 1, &sm.abort);
      if (!ok) break;
      tc::tmem_st32(scol, pk);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.p_full);
        // xbuf[xb] is read: P was computed from every value loaded from it, so
        // every lane's loads returned before its P store could issue
        mbar_arrive_cluster_relaxed(xfree_remote[xb]);  // the partner may send block gb + 2
      }
      const float2 s01 = add2(sum4[0], sum4[1]), s23 = add2(sum4[2], sum4[3]), s4 = add2(s01, s23);
      l += s4.x + s4.y;
      m = m_new;
    }
    if (!ok) break;
    // Epilogue: O / l -- bf16 output of an unsplit chunk, else the fp32
    // partial state; LSE in natural log (written by CTA 0 of the pair).
    ok = warp_wait(&sm.o_ready, nu & 1, &sm.abort);
    if (!ok) break;
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    const int64_t row = int64_t(u.b) * p.num_heads + r;
#pragma unroll 1
    for (int h = 0; h < kHalf / 32; ++h) {
      uint32_t ov[32];
      tc::tmem_ld32(tl + 32u * h, ov);
      tc::tmem_ld_wait();
      const int col = kHalf * int(rank) + 32 * h;
      if (row_ok && !sm.abort) {
        if (u.part < 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + row * kDc + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = tc::pack2<__nv_bfloat16>(__uint_as_float(ov[8 * q + 0]) * inv, __uint_as_float(ov[8 * q + 1]) * inv);
            v.y = tc::pack2<__nv_bfloat16>(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv);
            v.z = tc::pack2<__nv_bfloat16>(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv);
            v.w = tc::pack2<__nv_bfloat16>(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv);
            dst[q] = v;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.fws + p.partial_o_offset +
                                                  (int64_t(u.part) * kRows + r) * kDc + col);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(ov[4 * q]) * inv, __uint_as_float(ov[4 * q + 1]) * inv,
                                 __uint_as_float(ov[4 * q + 2]) * inv, __uint_as_float(ov[4 * q + 3]) * inv);
        }
      }
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.o_free);
    if (rank == 0 && row_ok && !sm.abort) {
      if (u.part < 0) {
        if (p.lse) p.lse[row] = lse_v;
      } else {
        p.fws[int64_t(u.part) * kRows + r] = lse_v;
      }
    }
    g += nb;
    ++nu;
  }
}

// Warps 8..11: thread r reads this CTA's partial logits of each block from
// TMEM (the same lanes as softmax thread r) as soon as S is complete, which is
// a block ahead of the softmax, and stores them asynchronously into the
// partner's xbuf; the bytes complete the partner's xfull.  The softmax of
// both CTAs then finds the other half already there.
__device__ void exchange_role(const Params& p, Smem& sm, uint32_t rank, int32_t begin, int32_t end,
                              int32_t off_units) {
  const int w = (threadIdx.x >> 5) - kExchangeWarp0;  // == warp % 4
  const int lane = threadIdx.x & 31;
  const int r = 32 * w + lane;
  const uint32_t tl = sm.tmem_base + (uint32_t(32 * w) << 16);
  const uint32_t peer = rank ^ 1u;
  const uint32_t x_remote[2] = {mapa_shared(smem_u32(&sm.xbuf[0][0][r]), peer),
                                mapa_shared(smem_u32(&sm.xbuf[1][0][r]), peer)};
  const uint32_t xfull_remote[2] = {mapa_shared(smem_u32(&sm.xfull[0]), peer),
                                    mapa_shared(smem_u32(&sm.xfull[1]), peer)};
  constexpr uint32_t kChunkStride = kRows * 16;  // bytes from chunk q to chunk q + 1 of a row
  int g = 0;
  bool ok = true;
  for (int32_t i = begin; i < end && ok; ++i) {
    const int nb = unit_blocks(load_unit(p.iws, off_units, i));
    for (int j = 0; j < nb; ++j) {
      const int gb = g + j, xb = gb & 1;
      ok = warp_wait(&sm.s_full[xb], (gb >> 1) & 1, &sm.abort);
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t sv[2][32];
      const uint32_t scol = tl + kTmemS + 64u * uint32_t(xb);
      tc::tmem_ld32(scol, sv[0]);
      tc::tmem_ld32(scol + 32, sv[1]);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_read[xb]);
      // the partner's softmax has read what was sent into this buffer for block gb - 2
      if (gb >= 2) {
        ok = warp_wait_cluster(&sm.xfree[xb], ((gb >> 1) - 1) & 1, &sm.abort);
        if (!ok) break;
      }
#pragma unroll
      for (int q = 0; q < kBlk / 4; ++q) {
        const uint32_t* v = &sv[q >> 3][4 * (q & 7)];
        st_async_v4(x_remote[xb] + kChunkStride * uint32_t(q), v[0], v[1], v[2], v[3], xfull_remote[xb]);
      }
    }
    g += nb;
  }
}

// ---------------------------------------------------------------- kernels

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ Params p) {
  // TMA/MMA operand blocks need a 1024-byte aligned base; a misaligned base
  // is reported instead of being used (both CTAs of a pair see the same).
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int32_t* iws = p.iws;
  const uint32_t rank = cluster_ctarank();
  const int32_t pair = int32_t(blockIdx.x >> 1);
  const int32_t n_units = __ldg(iws + FI_MLA_H_NUM_UNITS);
  const int32_t off_pair = __ldg(iws + FI_MLA_H_OFF_PAIR);
  bool bad = __ldg(iws + FI_MLA_H_MAGIC) != FI_MLA_MAGIC ||
             __ldg(iws + FI_MLA_H_NUM_PAIRS) != int32_t(gridDim.x >> 1) || (smem_u32(smem_raw) & 1023u) != 0;
  int32_t begin = 0, end = 0;
  if (!bad) {
    begin = __ldg(iws + off_pair + pair);
    end = __ldg(iws + off_pair + pair + 1);
    bad = begin < 0 || end < begin || end > n_units;
  }
  // The plan in the workspace must fit the buffers of this launch (a
  // workspace re-planned after the host checked the arguments is refused
  // here, before any write).
  if (!bad)
    bad = __ldg(iws + FI_MLA_H_NUM_PARTS) < 0 || __ldg(iws + FI_MLA_H_NUM_PARTS) > p.max_parts ||
          __ldg(iws + FI_MLA_H_BATCH) > p.q_rows || __ldg(iws + FI_MLA_H_NUM_HEADS) != p.num_heads ||
          __ldg(iws + FI_MLA_H_PAGE_SIZE) != p.page_size;
  if (bad) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPlan);
    return;
  }
  const int32_t off_units = __ldg(iws + FI_MLA_H_OFF_UNITS);
  const int32_t off_req = __ldg(iws + FI_MLA_H_OFF_REQ);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);   // the producer's arrive.expect_tx; TMA completes the bytes
      mbar_init(&sm.empty[s], 1);  // MMA commit
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_lat_full, 4);  // the four softmax warps
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.p_full, 4);      // the four softmax warps
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.o_ready, 1);
    mbar_init(&sm.o_free, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.xfull[b], 1);  // softmax thread 0's arrive.expect_tx; the partner's stores complete the bytes
      mbar_init(&sm.xfree[b], 4);  // the partner's four softmax warps
      mbar_init(&sm.s_read[b], 4); // this CTA's four exchange warps
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    // blocks 0 and 1 of the pair's stream land in xbuf 0 and 1
    mbar_arrive_expect_tx(&sm.xfull[0], kRows * kBlk * 4);
    mbar_arrive_expect_tx(&sm.xfull[1], kRows * kBlk * 4);
    fence_mbar_init();
  }
  if (warp == kAllocWarp) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the partner's barriers exist before anything arrives on them
  tc::fence_after_sync();

  if (warp == kProducerWarp) {
    producer(p, sm, rank, begin, end, off_units, off_req);
  } else if (warp == kMmaWarp) {
    mma_issuer(p, sm, begin, end, off_units);
  } else if (warp >= kExchangeWarp0) {
    exchange_role(p, sm, rank, begin, end, off_units);
  } else if (warp >= kSoftmaxWarp0) {
    softmax_role(p, sm, rank, begin, end, off_units);
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // no write of the partner into this CTA's shared memory is still on its way
  if (warp == kAllocWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(sm.tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(p.status, sm.abort);
}

// Merge of the chunks of split requests (the LSE-weighted combination of
// partial states), and (0, -inf) for requests with no cached token.  One warp
// per (merge entry, head) task, grid-stride; lane l holds dims 16l..16l+15,
// so each part's row is one coalesced 2 KB read per warp.  Nothing is merged
// when the decode kernel has set the status word (its partial states may be
// incomplete, or the plan may not fit this launch's buffers).
__global__ void __launch_bounds__(kMergeThreads) mla_merge_kernel(const int32_t* iws, const float* fws,
                                                                  int64_t partial_o_offset, uint16_t* o, float* lse,
                                                                  int32_t num_heads) {
  if (*reinterpret_cast<const volatile int32_t*>(iws + FI_MLA_H_STATUS) != 0) return;
  const int32_t n_merge = __ldg(iws + FI_MLA_H_NUM_MERGE);
  const int32_t off_merge = __ldg(iws + FI_MLA_H_OFF_MERGE);
  const int64_t tasks = int64_t(n_merge) * num_heads;
  const int lane = threadIdx.x & 31;
  constexpr int kWarps = kMergeThreads / 32;
  for (int64_t task = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); task < tasks;
       task += int64_t(gridDim.x) * kWarps) {
    const int32_t mi = int32_t(task / num_heads), h = int32_t(task - int64_t(mi) * num_heads);
    const int4 e = __ldg(reinterpret_cast<const int4*>(iws + off_merge) + mi);  // {b, part0, n_parts, 0}
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    float out_lse = -INFINITY;
    if (e.z > 0) {
      float M = -INFINITY;
      for (int k = lane; k < e.z; k += 32) M = fmaxf(M, __ldg(fws + int64_t(e.y + k) * kRows + h));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
      float L = 0.f;
      for (int k = 0; k < e.z; ++k) {
        const float s = __ldg(fws + int64_t(e.y + k) * kRows + h);
        const float wgt = M == -INFINITY ? 0.f : expf(s - M);
        const float4* v =
            reinterpret_cast<const float4*>(fws + partial_o_offset + (int64_t(e.y + k) * kRows + h) * kDc) + 4 * lane;
        float4 x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = __ldg(v + q);
        L += wgt;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[4 * q] += wgt * x[q].x;
          acc[4 * q + 1] += wgt * x[q].y;
          acc[4 * q + 2] += wgt * x[q].z;
          acc[4 * q + 3] += wgt * x[q].w;
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] *= inv;
      out_lse = L > 0.f ? M + logf(L) : -INFINITY;
    }
    const int64_t row = int64_t(e.x) * num_heads + h;
    uint4 pk[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      pk[q].x = tc::pack2<__nv_bfloat16>(acc[8 * q], acc[8 * q + 1]);
      pk[q].y = tc::pack2<__nv_bfloat16>(acc[8 * q + 2], acc[8 * q + 3]);
      pk[q].z = tc::pack2<__nv_bfloat16>(acc[8 * q + 4], acc[8 * q + 5]);
      pk[q].w = tc::pack2<__nv_bfloat16>(acc[8 * q + 6], acc[8 * q + 7]);
    }
    uint4* dst = reinterpret_cast<uint4*>(o + row * kDc) + 2 * lane;
    dst[0] = pk[0];
    dst[1] = pk[1];
    if (lse && lane == 0) lse[row] = out_lse;
  }
}

// Shared-memory opt-in of the decode kernel, once per device.
constexpr int kMaxDevices = 64;
cudaError_t configure(int dev) {
  static bool done[kMaxDevices] = {};
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return e;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool stride_ok(int64_t elems) { return elems > 0 && (elems * 2) % 16 == 0; }

}  // namespace mla
}  // namespace fi

using namespace fi;
using namespace fi::mla;

extern "C" fi_status fi_mla_default_config(int device, fi_mla_config* out) {
  if (!out) return FI_ERR_INVALID_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return FI_ERR_CUDA;
  int clusters = 0;
  cudaError_t e = configure(device);
  if (e == cudaSuccess) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3(unsigned(2 * (sms > 0 ? sms : 2)), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = kSmemBytes;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, mla_decode_kernel, &lc);
  }
  cudaSetDevice(prev);
  if (e != cudaSuccess || clusters < 1) return FI_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  out->num_pairs = clusters;
  out->max_batch = 4096;
  out->max_units = 1 << 15;
  out->max_parts = 512;
  out->min_chunk = 256;
  return FI_OK;
}

extern "C" fi_status fi_mla_decode_run(const fi_mla_plan_info* info, const void* q_nope, int64_t q_nope_stride_tok,
                                       int64_t q_nope_stride_head, const void* q_pe, int64_t q_pe_stride_tok,
                                       int64_t q_pe_stride_head, int32_t q_rows, const void* ckv,
                                       int64_t ckv_stride_page, int64_t ckv_stride_slot, const void* kpe,
                                       int64_t kpe_stride_page, int64_t kpe_stride_slot, int32_t num_pages,
                                       const int32_t* kv_indices_dev, void* o, float* lse, float sm_scale,
                                       void* int_workspace_dev, void* float_workspace_dev, void* stream) {
  if (!info || !q_nope || !q_pe || !ckv || !kpe || !kv_indices_dev || !o || !int_workspace_dev)
    return FI_ERR_INVALID_ARG;
  if (info->num_pairs < 1 || q_rows < 1 || q_rows < info->batch || num_pages < 1 || !std::isfinite(sm_scale))
    return FI_ERR_INVALID_ARG;
  if (info->num_parts > 0 && !float_workspace_dev) return FI_ERR_INVALID_ARG;
  const int H = info->num_heads, P = info->page_size;
  if (H < 1 || H > kRows) return FI_ERR_UNSUPPORTED;
  if (P != 8 && P != 16 && P != 32 && P != 64) return FI_ERR_UNSUPPORTED;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(ckv) || !aligned16(kpe) || !aligned16(o) ||
      !aligned16(int_workspace_dev) || (float_workspace_dev && !aligned16(float_workspace_dev)) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FI_ERR_ALIGNMENT;
  if (!stride_ok(q_nope_stride_tok) || !stride_ok(q_nope_stride_head) || !stride_ok(q_pe_stride_tok) ||
      !stride_ok(q_pe_stride_head) || !stride_ok(ckv_stride_page) || !stride_ok(ckv_stride_slot) ||
      !stride_ok(kpe_stride_page) || !stride_ok(kpe_stride_slot))
    return FI_ERR_ALIGNMENT;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure(dev) != cudaSuccess) return FI_ERR_CUDA;
  Params p;
  std::memset(&p, 0, sizeof p);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t qp_d[3] = {uint64_t(FI_MLA_ROPE_DIM), uint64_t(H), uint64_t(q_rows)};
  const int64_t qp_s[2] = {q_pe_stride_head, q_pe_stride_tok};
  const uint32_t qp_b[3] = {uint32_t(kRopeHalf), uint32_t(kRows), 1u};
  const uint64_t ckv_d[3] = {uint64_t(kDc), uint64_t(P), uint64_t(num_pages)};
  const int64_t ckv_s[2] = {ckv_stride_slot, ckv_stride_page};
  const uint64_t kpe_d[3] = {uint64_t(FI_MLA_ROPE_DIM), uint64_t(P), uint64_t(num_pages)};
  const int64_t kpe_s[2] = {kpe_stride_slot, kpe_stride_page};
  const uint32_t ckv_b[3] = {64u, uint32_t(P), 1u};
  const uint32_t kpe_b[3] = {uint32_t(kRopeHalf), uint32_t(P), 1u};
  if (!make_map(&p.tm_qp, bf, q_pe, 3, qp_d, qp_s, qp_b, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&p.tm_ckv, bf, ckv, 3, ckv_d, ckv_s, ckv_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tm_kpe, bf, kpe, 3, kpe_d, kpe_s, kpe_b, CU_TENSOR_MAP_SWIZZLE_64B))
    return FI_ERR_UNSUPPORTED;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.qn_stride_tok = q_nope_stride_tok;
  p.qn_stride_head = q_nope_stride_head;
  p.iws = static_cast<const int32_t*>(int_workspace_dev);
  p.status = static_cast<int32_t*>(int_workspace_dev) + FI_MLA_H_STATUS;
  p.kv_indices = kv_indices_dev;
  p.fws = static_cast<float*>(float_workspace_dev);
  p.partial_o_offset = fi_mla_partial_o_offset(info->max_parts > 0 ? info->max_parts : 1);
  p.max_parts = p.fws ? info->max_parts : 0;
  p.q_rows = q_rows;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.num_heads = H;
  p.page_size = P;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = 2 * info->num_pairs;
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return FI_ERR_CUDA;
  // the merge reads each partial state once: enough blocks to keep several
  // tasks' loads in flight per SM (the count of tasks is known on the device)
  mla_merge_kernel<<<kMergeBlocksPerPair * info->num_pairs, kMergeThreads, 0, s>>>(p.iws, p.fws, p.partial_o_offset,
                                                                                   p.o, lse, H);
  e = cudaGetLastError();
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}
