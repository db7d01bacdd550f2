// run_bf16_rope.cu -- bf16 run kernels with RoPE fused into the loaders, with
// and without a logits soft-cap and a sliding-window / sink mask.
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__nv_bfloat16, false, false, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__nv_bfloat16, true, false, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__nv_bfloat16, false, true, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__nv_bfloat16, true, true, true>(const RunParams&, int, cudaStream_t);

}  // namespace fi
