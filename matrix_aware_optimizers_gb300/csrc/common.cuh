// Shared device/host helpers of libmao (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mao.h"

namespace mao {

// ---------------------------------------------------------------- host helpers

// Bytes per element (MAO_SIGN1 is addressed by 4-byte words).
inline int elem_size(int32_t dt) { return dt == MAO_BF16 ? 2 : dt == MAO_I8 ? 1 : 4; }
inline bool valid_dtype(int32_t dt) { return dt == MAO_F32 || dt == MAO_BF16; }

// Checks a descriptor: non-null data, positive sizes, ld >= cols, element alignment.
inline mao_status check_mat(const mao_mat& m, bool allow_null_data = false) {
  if (!valid_dtype(m.dtype) || m.reserved != 0) return MAO_ERR_INVALID_ARG;
  if (m.rows < 1 || m.cols < 1 || m.ld < m.cols) return MAO_ERR_INVALID_ARG;
  if (m.rows > (int64_t(1) << 31) || m.cols > (int64_t(1) << 31)) return MAO_ERR_UNSUPPORTED;
  if (m.data == nullptr) return allow_null_data ? MAO_OK : MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(m.data) % elem_size(m.dtype) != 0) return MAO_ERR_MISALIGNED;
  return MAO_OK;
}

// Checks an ns_orthogonalize input: f32/bf16 as check_mat, or an int8 / packed sign matrix
// (the optional polar step on an aggregated sign matrix).
inline mao_status check_ns_input(const mao_mat& m) {
  if (m.dtype != MAO_I8 && m.dtype != MAO_SIGN1) return check_mat(m);
  if (m.reserved != 0 || m.rows < 1 || m.cols < 1 || m.ld < m.cols) return MAO_ERR_INVALID_ARG;
  if (m.rows > (int64_t(1) << 31) || m.cols > (int64_t(1) << 31)) return MAO_ERR_UNSUPPORTED;
  if (m.dtype == MAO_SIGN1 && m.ld != m.cols) return MAO_ERR_INVALID_ARG;
  if (m.data == nullptr) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(m.data) % elem_size(m.dtype) != 0) return MAO_ERR_MISALIGNED;
  return MAO_OK;
}

// True when rows of 8 elements can be moved with 16-byte vector accesses.
inline bool vec8_ok(const mao_mat& m) {
  const int es = elem_size(m.dtype);
  return (reinterpret_cast<uintptr_t>(m.data) % 16 == 0) && (m.cols % 8 == 0) &&
         ((m.ld * es) % 16 == 0);
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

inline mao_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MAO_OK : MAO_ERR_CUDA; }

// Number of SMs of the current device (cached per device id).
int num_sms();
// Compute capability major*10+minor of the current device (cached).
int device_cc();

// -------------------------------------------------------------- device helpers

struct alignas(16) bf16x8 { __nv_bfloat162 h[4]; };

__device__ __forceinline__ float load_elem(const void* p, int64_t idx, int32_t dt) {
  return dt == MAO_BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx])
                        : reinterpret_cast<const float*>(p)[idx];
}

__device__ __forceinline__ void store_elem(void* p, int64_t idx, int32_t dt, float v) {
  if (dt == MAO_BF16) reinterpret_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(p)[idx] = v;
}

// Loads 8 consecutive elements (16-byte aligned address) as fp32.
__device__ __forceinline__ void load8(const void* p, int64_t idx, int32_t dt, float (&v)[8]) {
  if (dt == MAO_BF16) {
    const uint4 raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p) + idx);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + idx);
    const float4 a = q[0], b = q[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Stores 8 consecutive fp32 values (16-byte aligned address), rounding to dt.
__device__ __forceinline__ void store8(void* p, int64_t idx, int32_t dt, const float (&v)[8]) {
  if (dt == MAO_BF16) {
    uint4 raw;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p) + idx) = raw;
  } else {
    float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(p) + idx);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

}  // namespace mao
