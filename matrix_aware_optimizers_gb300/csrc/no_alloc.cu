// ns_orthogonalize_noalloc: Newton–Schulz with a library-owned, statically sized scratch
// area instead of a caller-provided workspace.
//
// Some callers cannot call cudaMalloc: code that runs inside a host framework that owns all
// device memory through its own pool and forbids allocations behind its back, or a
// latency-critical loop that must never pay cudaMalloc's implicit device synchronisation.
// For them this entry point takes only inputs and outputs; its scratch lives in one
// file-scope __device__ array that every GPU loading this library holds until the process
// exits.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mao {
namespace {

// The scratch area (MAO_NOALLOC_WORKSPACE_BYTES bytes, 256-byte aligned), shared by every
// call on a device. In host code this name is only a stand-in for the symbol; the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MAO_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch area on the current device. Outside stream capture it is
// looked up on every call: after a cudaDeviceReset, or in another context on the same
// device, the module is loaded again and the array may sit at another address. During a
// capture the address of the last lookup on this device is used (a capture must not be the
// first use of the call on a device, nor the first use after a reset).
mao_status scratch_address(cudaStream_t stream, void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MAO_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MAO_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MAO_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (g_scratch_ptr[dev] == nullptr) {
    return MAO_ERR_UNSUPPORTED;  // first use on this device inside a capture
  }
  *ptr = g_scratch_ptr[dev];
  return MAO_OK;
}

}  // namespace
}  // namespace mao

using namespace mao;

extern "C" size_t ns_noalloc_workspace_bytes(void) { return size_t(MAO_NOALLOC_WORKSPACE_BYTES); }

extern "C" mao_status ns_orthogonalize_noalloc(const mao_mat* in, const mao_mat* out,
                                               int32_t batch, int32_t steps,
                                               const float* coeffs, int32_t coeff_stride,
                                               float eps, int32_t compute,
                                               uint32_t* const* sign_bits, void* stream) {
  // Same argument rules as ns_orthogonalize.
  if (!in || !out || batch < 1 || steps < 1 || steps > 64 || !coeffs) return MAO_ERR_INVALID_ARG;
  if (coeff_stride != 0 && coeff_stride != 3) return MAO_ERR_INVALID_ARG;
  if (!valid_dtype(compute) || !std::isfinite(eps) || eps < 0.0f) return MAO_ERR_INVALID_ARG;
  for (int i = 0; i < (coeff_stride ? 3 * steps : 3); ++i)
    if (!std::isfinite(coeffs[i])) return MAO_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_ns_input(in[b]);
    if (st != MAO_OK) return st;
    const bool bits = sign_bits && sign_bits[b];
    st = check_mat(out[b], bits);
    if (st != MAO_OK) return st;
    if (out[b].rows != in[b].rows || out[b].cols != in[b].cols) return MAO_ERR_INVALID_ARG;
    if (bits && (reinterpret_cast<uintptr_t>(sign_bits[b]) % 4 != 0)) return MAO_ERR_MISALIGNED;
  }
  // The batch must fit the fixed scratch area; larger requests are refused before any
  // device work (use ns_orthogonalize with a caller-provided workspace instead).
  const size_t need = ns_workspace_size(in, batch, compute);
  if (need > size_t(MAO_NOALLOC_WORKSPACE_BYTES)) return MAO_ERR_WORKSPACE;
  if (compute == MAO_BF16 && device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const mao_status st = scratch_address(static_cast<cudaStream_t>(stream), &scratch);
  if (st != MAO_OK) return st;
  // Nothing in the scratch area has to start at zero: every region the products read is
  // written earlier in the same call (staged inputs, norms, A, B, X), so the contents a
  // previous call left behind are never used.
  return ns_run(in, out, batch, steps, coeffs, coeff_stride, eps, compute, sign_bits, scratch,
                size_t(MAO_NOALLOC_WORKSPACE_BYTES), static_cast<cudaStream_t>(stream));
}
