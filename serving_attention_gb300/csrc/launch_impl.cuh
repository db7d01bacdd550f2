// launch_impl.cuh -- definition of launch_run; included by the translation
// units that instantiate it (run_*.cu), each for a few kernel variants.
#pragma once
#include <cuda_runtime.h>

#include "attention_kernel.cuh"
#include "launch.h"

namespace fi {

// The shared-memory opt-in is set once per device and instantiation, so a
// run enqueued inside a stream capture makes no non-stream CUDA call.
template <typename T, bool kCap, bool kMask, bool kRope>
cudaError_t launch_run(const RunParams& p, int num_ctas, cudaStream_t stream) {
  static bool configured[kMaxDevices] = {};
  auto kern = paged_attention_kernel<T, kCap, kMask, kRope>;
  const int smem = int(kSmemBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !configured[dev]) {
    // The tensor-core phase moves registers between warpgroups; that needs the
    // launch to hold at least kRegsLaunch registers per thread.
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) configured[dev] = true;
  }
  kern<<<num_ctas, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fi
