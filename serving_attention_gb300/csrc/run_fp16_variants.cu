// run_fp16_variants.cu -- fp16 run kernels with a logits soft-cap and/or a
// sliding-window / sink mask.
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__half, true, false, false>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__half, false, true, false>(const RunParams&, int, cudaStream_t);
template cudaError_t launch_run<__half, true, true, false>(const RunParams&, int, cudaStream_t);

}  // namespace fi
