// ptx.cuh -- thin inline-PTX wrappers (mbarrier, cp.async, named barriers,
// bounded waits) shared by the kernels of this library.  sm_103a only.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fi {

// Device status bits, OR-ed into the int workspace's status word
// (kStatusRange: a value rotated into fp16 left the fp16 range).
enum : int32_t { kStatusTimeout = 1, kStatusBadPlan = 2, kStatusRange = 4 };

// A bounded wait gives up after this many SM clocks (about half a second at
// 2 GHz) and reports kStatusTimeout instead of hanging the GPU.
constexpr long long kWaitBudgetClocks = 1000000000LL;
constexpr int kPollsPerCheck = 8;  // polls of a warp-wide wait between checks of the abort flag and the budget

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware until the phase
// completes or about kSuspendHintNs nanoseconds pass, instead of spinning:
// a waiting warp then takes no issue slots from the warps that compute.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking: has the phase with `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Warp-uniform bounded wait, called by a converged warp.  Every lane polls
// (a branch around a single polling lane costs more than the poll itself);
// lane 0's view of completion, abort and budget is broadcast, so all lanes
// leave on the same iteration with the same result: false when the budget ran
// out (the abort flag is then set) or another role gave up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  // Fast path: one poll, no read of the abort flag (a shared-memory read is
  // slow while the tensor core streams its operands from shared memory).
  if (__shfl_sync(0xffffffffu, mbar_try_wait(bar, parity) ? 1 : 0, 0)) return true;
  const long long t0 = clock64();
  while (true) {
    // a few polls between the checks of the abort flag and the budget
#pragma unroll 1
    for (int k = 0; k < kPollsPerCheck; ++k)
      if (__shfl_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity) ? 1 : 0, 0)) return true;
    const int gave_up = *abort != 0 ? 2 : 0;
    const int late = clock64() - t0 > kWaitBudgetClocks ? 4 : 0;
    const int st = __shfl_sync(0xffffffffu, gave_up | late, 0);
    if (st & 2) return false;
    if (st & 4) {
      *abort = kStatusTimeout;  // every lane stores the same value
      return false;
    }
  }
}

// Warp-uniform bounded wait for up to four barrier phases at once: lane l
// polls entry l (lanes past n repeat entry 0), so one instruction covers the
// whole list.  Same results and abort behaviour as warp_wait.
__device__ __forceinline__ bool warp_wait_all(int n, uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                              uint64_t* b2, uint32_t p2, uint64_t* b3, uint32_t p3,
                                              volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const int e = lane < n ? lane : 0;
  uint64_t* bar = e == 0 ? b0 : e == 1 ? b1 : e == 2 ? b2 : b3;
  const uint32_t parity = e == 0 ? p0 : e == 1 ? p1 : e == 2 ? p2 : p3;
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < kPollsPerCheck; ++k)
      if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity))) return true;
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

// Bounded wait that ignores the abort flag: used to drain a role's own
// asynchronous copies or MMAs before the CTA leaves.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitBudgetClocks) return;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 16-byte async copy global -> shared; src_bytes = 0 writes 16 zero bytes.
__device__ __forceinline__ void cp_async_16(void* dst_smem, const void* src_gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src_gmem),
               "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count must include this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// The same barrier reached from different places in the code (barrier.sync
// without .aligned): the roles of a CTA meet here from their own branches.
__device__ __forceinline__ void named_barrier_sync_unaligned(uint32_t id, uint32_t threads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Packed fp32 fused multiply-add of two lanes at once: a * b + c per lane,
// each rounded once (sm_100 and later).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&r);
}

// Packed fp32 add of two lanes at once (sm_100 and later).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<const float2*>(&r);
}

// Three-input maximum (sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element conversions of 16-bit storage types.
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  __device__ __forceinline__ static float2 to_float2(uint32_t packed) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&packed));
  }
  __device__ __forceinline__ static uint32_t from_float2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

template <>
struct Elem<__half> {
  __device__ __forceinline__ static float2 to_float2(uint32_t packed) {
    return __half22float2(*reinterpret_cast<const __half2*>(&packed));
  }
  __device__ __forceinline__ static uint32_t from_float2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// Programmatic dependent launch: a merge that follows a kernel is enqueued
// with programmatic stream serialization, and that kernel lets its
// dependents be scheduled from its start (`let_dependents_start`), so the
// merge's blocks take SMs as the kernel's CTAs leave instead of after the
// whole grid has finished and a new launch has gone through; each waits in
// `grid_dependency_wait` until the preceding grid has completed and its
// memory is visible (launched without the attribute, the wait returns at
// once).
__device__ __forceinline__ void let_dependents_start() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_behind_run(void (*kernel)(KArgs...), int32_t blocks, int threads, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, KArgs(args)...);
}


}  // namespace fi
