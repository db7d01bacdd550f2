// run_fp16.cu -- the plain fp16 run kernel (no logits cap, no window mask).
#include "launch_impl.cuh"

namespace fi {

template cudaError_t launch_run<__half, false, false, false>(const RunParams&, int, cudaStream_t);

}  // namespace fi
