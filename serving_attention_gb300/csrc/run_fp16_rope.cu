// run_fp16_rope.cu -- fp16 run kernels with RoPE fused into the loaders, with
// and without a logits soft-cap and a sliding-window / sink mask.
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__half, false, false, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__half, true, false, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__half, false, true, true>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__half, true, true, true>(const RunParams&, int, cudaStream_t);

}  // namespace fi
