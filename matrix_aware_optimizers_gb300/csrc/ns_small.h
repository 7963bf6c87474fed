// Newton–Schulz of small matrices on the fp32 accuracy path in one launch (ns_small.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mao.h"

namespace mao {

constexpr int kSmallMaxPerLaunch = 64;          // matrices per launch (one cluster each)
constexpr size_t kSmallSmemMax = 200 * 1024;    // shared memory of one CTA of the cluster

// Shared memory one CTA needs for an R x C matrix (SIZE_MAX when far too large).
size_t ns_small_smem_bytes(int64_t R, int64_t C);
// True when every matrix of the call can take the one-launch path: fp32 compute, f32 or
// bf16 inputs and outputs, and each matrix's working set within kSmallSmemMax.
bool ns_small_eligible(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                       int32_t compute);
// The whole Newton–Schulz call (normalisation, every iteration, U and packed signs). With G,
// the momentum M <- fma(mu, M, G) (rounded to M's dtype) comes first in the same launch:
// `in` holds M, which the call updates in place, and the iteration starts from the new M.
mao_status ns_small_run(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                        const float* coeffs, int32_t coeff_stride, float eps,
                        uint32_t* const* sign_bits, cudaStream_t stream,
                        const mao_mat* G = nullptr, float mu = 0.0f);
// Reads and clears the small kernel's error word (a row exchange that timed out).
mao_status small_read_and_clear_error(cudaStream_t stream);

}  // namespace mao
