// Blockwise Newton–Schulz: every block of a fixed grid over each matrix is orthogonalised
// on its own, as each rank of the blockwise mode does with the block of the momentum it
// owns ("NVIDIA MegatronによるLLM学習高速化へ向けた新世代オプティマイザの高度化", section
// 分散モード, blockwise paragraph). Host code only: the blocks become strided descriptors of
// one grouped ns_run call (equal block shapes share a group), so no block is copied out.
#include <algorithm>
#include <cmath>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mao {
namespace {

constexpr int64_t kMaxBlocks = int64_t(1) << 20;

// Strided descriptor of block (i0, j0) of m.
mao_mat block_of(const mao_mat& m, int64_t i0, int64_t j0, int64_t br, int64_t bc) {
  mao_mat b = m;
  if (m.data)
    b.data = static_cast<char*>(m.data) + (i0 * m.ld + j0) * int64_t(elem_size(m.dtype));
  b.rows = std::min(br, m.rows - i0);
  b.cols = std::min(bc, m.cols - j0);
  return b;
}

mao_status expand(const mao_mat* X, const mao_mat* Y, int32_t batch, int64_t br, int64_t bc,
                  std::vector<mao_mat>& bx, std::vector<mao_mat>* by) {
  if (!X || batch < 1 || br < 1 || bc < 1) return MAO_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) {
    if (X[b].rows < 1 || X[b].cols < 1) return MAO_ERR_INVALID_ARG;
    total += ceil_div(X[b].rows, br) * ceil_div(X[b].cols, bc);
    if (total > kMaxBlocks) return MAO_ERR_UNSUPPORTED;
  }
  bx.clear();
  bx.reserve(size_t(total));
  if (by) {
    by->clear();
    by->reserve(size_t(total));
  }
  for (int b = 0; b < batch; ++b)
    for (int64_t i0 = 0; i0 < X[b].rows; i0 += br)
      for (int64_t j0 = 0; j0 < X[b].cols; j0 += bc) {
        bx.push_back(block_of(X[b], i0, j0, br, bc));
        if (by) by->push_back(block_of(Y[b], i0, j0, br, bc));
      }
  return MAO_OK;
}

}  // namespace
}  // namespace mao

using namespace mao;

extern "C" {

size_t ns_blockwise_workspace_bytes(const mao_mat* X, int32_t batch, int64_t block_rows,
                                    int64_t block_cols, int32_t compute) {
  if (!valid_dtype(compute)) return 0;
  std::vector<mao_mat> bx;
  if (expand(X, nullptr, batch, block_rows, block_cols, bx, nullptr) != MAO_OK) return 0;
  for (const auto& m : bx)
    if (m.rows > (int64_t(1) << 31) || m.cols > (int64_t(1) << 31)) return 0;
  return ns_workspace_size(bx.data(), int32_t(bx.size()), compute);
}

mao_status ns_orthogonalize_blockwise(const mao_mat* in, const mao_mat* out, int32_t batch,
                                      int64_t block_rows, int64_t block_cols, int32_t steps,
                                      const float* coeffs, int32_t coeff_stride, float eps,
                                      int32_t compute, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  if (!in || !out || batch < 1 || steps < 1 || steps > 64 || !coeffs) return MAO_ERR_INVALID_ARG;
  if (block_rows < 1 || block_cols < 1) return MAO_ERR_INVALID_ARG;
  if (coeff_stride != 0 && coeff_stride != 3) return MAO_ERR_INVALID_ARG;
  if (!valid_dtype(compute) || !std::isfinite(eps) || eps < 0.0f) return MAO_ERR_INVALID_ARG;
  for (int i = 0; i < (coeff_stride ? 3 * steps : 3); ++i)
    if (!std::isfinite(coeffs[i])) return MAO_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    // packed signs have no row stride, so they cannot be cut into strided blocks
    if (in[b].dtype == MAO_SIGN1) return MAO_ERR_INVALID_ARG;
    mao_status st = check_ns_input(in[b]);
    if (st == MAO_OK) st = check_mat(out[b]);
    if (st != MAO_OK) return st;
    if (out[b].rows != in[b].rows || out[b].cols != in[b].cols) return MAO_ERR_INVALID_ARG;
  }
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (compute == MAO_BF16 && device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  std::vector<mao_mat> bi, bo;
  mao_status st = expand(in, out, batch, block_rows, block_cols, bi, &bo);
  if (st != MAO_OK) return st;
  const int32_t nb = int32_t(bi.size());
  if (workspace_bytes < ns_workspace_size(bi.data(), nb, compute)) return MAO_ERR_WORKSPACE;
  return ns_run(bi.data(), bo.data(), nb, steps, coeffs, coeff_stride, eps, compute, nullptr,
                workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
