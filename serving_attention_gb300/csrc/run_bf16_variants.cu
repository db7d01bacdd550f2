// run_bf16_variants.cu -- bf16 run kernels with a logits soft-cap and/or a
// sliding-window / sink mask.
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__nv_bfloat16, true, false, false>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__nv_bfloat16, false, true, false>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__nv_bfloat16, true, true, false>(const RunParams&, int, cudaStream_t);

}  // namespace fi
