// Launcher of the two-state merge kernel (csrc/merge.cu).
#pragma once
#include <cuda_runtime.h>

namespace mla {

// Two attention states of `rows` rows (fp32 [rows, 512] + lse [rows]) into
// one (bf16 or fp32 [rows, 512] + lse [rows]); the outputs may alias inputs.
cudaError_t launch_merge_states(const float* o_a, const float* lse_a, const float* o_b,
                                const float* lse_b, void* out, bool out_f32, float* lse_out,
                                int rows, cudaStream_t s);

}  // namespace mla
