// Internal launch interface of the LSE merge (merge.cu) for the C ABI (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace paq8 {

cudaError_t launch_merge_states(const uint16_t *out_a, const float *lse_a, const uint16_t *out_b,
                                const float *lse_b, uint16_t *out, float *lse, int64_t num_rows,
                                int32_t d, cudaStream_t stream);

}  // namespace paq8
