// run_bf16.cu -- the plain bf16 run kernel (no logits cap, no window mask).
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__nv_bfloat16, false, false, false>(const RunParams&, int, cudaStream_t);

cudaError_t run_kernel_occupancy(int* per_sm) {
  auto kern = paged_attention_kernel<__nv_bfloat16, false, false, false>;
  const int smem = int(kSmemBytes);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, kThreads, smem);
  return e;
}

}  // namespace fi
