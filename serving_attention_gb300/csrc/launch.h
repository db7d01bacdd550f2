// launch.h -- launches of the persistent run kernel, one explicit
// instantiation per element type and variant (logits soft-cap kCap, sliding
// window / sink mask kMask, RoPE kRope), spread over several translation
// units so that they compile in parallel.
#pragma once
#include <cuda_runtime.h>

#include "attention.cuh"

namespace fi {

constexpr int kMaxDevices = 64;  // devices with per-device launch state

// Enqueues paged_attention_kernel<T, kCap, kMask, kRope> on `stream` with the
// plan's grid.  Refuses (cudaErrorInvalidConfiguration) a build whose
// register count cannot cover the tensor-core phase's register split.
template <typename T, bool kCap, bool kMask, bool kRope>
cudaError_t launch_run(const RunParams& p, int num_ctas, cudaStream_t stream);

// Resident CTAs per SM of the plain bf16 kernel (the occupancy the plan's
// default grid is sized by); sets the kernel's shared-memory opt-in.
cudaError_t run_kernel_occupancy(int* per_sm);

}  // namespace fi
