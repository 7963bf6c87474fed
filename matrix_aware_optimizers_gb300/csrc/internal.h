// Internal launchers behind the C ABI (arguments already validated by abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mao.h"

namespace mao {

mao_status momentum_launch(const mao_mat* M, const mao_mat* G, int32_t batch, float mu,
                           cudaStream_t stream);
mao_status update_launch(const mao_mat* W, const uint32_t* const* vote, const mao_mat* U,
                         int32_t batch, float lr, cudaStream_t stream);
mao_status sign_pack_launch(const mao_mat& U, uint32_t* bits, cudaStream_t stream);
mao_status sign_int8_launch(const mao_mat& U, int8_t* s, cudaStream_t stream);
mao_status vote_int8_launch(const int8_t* s, int32_t n_workers, int64_t stride, int64_t n,
                            int8_t* sum, int8_t* sbar, uint32_t* vote, cudaStream_t stream);
// Vote and Sign-Muon update of W in one launch (the words of vote_launch, then
// W <- W - lr * (+1 / -1) as update_launch with a vote).
mao_status vote_update_launch(const uint32_t* bits, int32_t n_workers, int64_t stride,
                              int64_t nbits, uint32_t* vote, const mao_mat& W, float lr,
                              cudaStream_t stream);
mao_status vote_launch(const uint32_t* bits, int32_t n_workers, int64_t stride, int64_t nbits,
                       uint32_t* vote, cudaStream_t stream);

size_t ns_workspace_size(const mao_mat* X, int32_t batch, int32_t compute);
// A whole Muon step around Newton–Schulz (muon_step): the staging pass first sets
// in[b] <- fmaf(mu, in[b], G[b]) (rounded to its dtype) and orthogonalises the new values;
// with update set, the last product then updates out[b] <- out[b] - lr * U in place instead
// of writing U (without it the call's outputs are as without the momentum: U or its signs).
struct NsFuse {
  const mao_mat* G;
  const mao_mat* W_in;  // null: out[b] is updated in place; else out[b] <- W_in[b] - lr * U
  float mu, lr;
  bool update = true;
};
mao_status ns_run(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                  const float* coeffs, int32_t coeff_stride, float eps, int32_t compute,
                  uint32_t* const* sign_bits, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream, const NsFuse* fuse = nullptr);

// Bound of every device-side wait in the tensor-core kernels (mao_set_wait_limit).
unsigned long long wait_limit_ns();

// Launch accounting (every kernel launch of the library calls this once).
void count_launch();
// Optional timing of launches (see mao_profile_begin); tag 0 = tensor-core product kernel,
// other tags name the Dion CUDA-core kernels (mao_profile_end_tagged).
void profile_before_launch(cudaStream_t stream, int tag = 0);
void profile_after_launch(cudaStream_t stream);
// Optional timing of whole runs of tensor-core products (mao_profile_span_begin): one event
// before the first product of a Newton–Schulz call and one after its last, so the products
// keep overlapping one another's set-up (programmatic dependent launch) while timed.
void profile_span_begin(cudaStream_t stream);
void profile_span_end(cudaStream_t stream);

// Reads and clears the device error word of the tensor-core kernels (after a stream sync).
mao_status tc_read_and_clear_error(cudaStream_t stream);
// Reads and clears the Cholesky pivot error word of the Dion kernels.
mao_status dion_read_and_clear_error(cudaStream_t stream);

// Entry in the workspace table of final outputs, one per matrix slot.
struct OutEntry {
  void* out;        // U destination (may be null)
  uint32_t* bits;   // packed signs destination (may be null)
  int64_t ld;       // U row stride (elements)
  int32_t dtype;    // U dtype
  int32_t flags;    // bit 0: 16-byte vector stores allowed; bit 1: one sign word per 32 columns
  const void* src;  // in-place updates (TC_UPDATE): the old values, of out's dtype, or null
                    // for out itself (out <- src + a (A B^T))
  int64_t src_ld;   // row stride of src (elements)
  float* copy;      // optional fp32 copy of the first copy_cols columns (final products)
  int32_t copy_ld;  // row stride of copy (elements)
  int32_t copy_cols;
};

// OUT_COPY_VEC: copy's rows allow 16-byte stores.
enum OutFlags : int32_t { OUT_VEC = 1, OUT_WORDS = 2, OUT_COPY_VEC = 4 };

}  // namespace mao
