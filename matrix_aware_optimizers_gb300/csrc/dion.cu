// One Dion step on the GPU ("대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습",
// algorithm section): for each parameter matrix X (m x n) with momentum M, gradient G and
// the previous right factor Q (n x r),
//
//   B = M + G                       stage kernel: M <- B in place, bf16 copy Bw
//   P = orthonormalise(B Q)         tensor-core product (fp32 P), then Cholesky QR twice
//   R = B^T P                       tensor-core product (fp32 R)
//   Q <- ColumnNormalize(R)         column norms, then Q (fp32, caller) and bf16 copies
//   M <- B - (1 - mu) P R^T         tensor-core rank-r update, in place
//   X <- X - lr P Q^T               tensor-core rank-r update, in place
//
// The orthonormal basis is the Q factor of the thin QR with a positive triangular
// diagonal, computed as Cholesky QR applied twice: S = P^T P, S = L L^T, P <- P L^-T.
// The three dense products run on the same tcgen05 kernel as Newton–Schulz; the small
// r x r work (Gram matrices, Cholesky, triangular inverse) runs in fp32 on CUDA cores.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "ns_plan.h"

namespace mao {

__device__ unsigned int g_dion_error;  // bit 0: a Cholesky pivot was not positive

namespace {

constexpr int kChunk = 32;        // matrices per launch of the CUDA-core kernels
constexpr int kGramRows = 1024;   // rows of P summed by one partial Gram tile
constexpr int kMaxRank = 256;

struct DionMat {
  void* M;
  const void* G;
  void* X;
  float* Q;
  float* Pout;          // optional copy of the final P (m x r, row stride r)
  int64_t ldm, ldg, ldx, ldq;
  int32_t dtm, dtg, dtx;
  int32_t flags_m, flags_x;  // OutEntry flags of M and X (16-byte vector access allowed)
};

struct DionDims {
  int64_t m, n, r, ldn, ldr, nchunks;
};

struct DionBuf {
  __nv_bfloat16 *Bw, *Qw, *Rw, *Pw;  // bf16 operands: [count][m|n][ldn|ldr]
  float *P0, *P1, *Rf;               // fp32 [count][m|n][ldr]
  float *S, *Linv, *cn;              // [count][nchunks][r][r], [count][r][r], [count][r]
  OutEntry *tP, *tR, *tM, *tX;       // output tables of the tensor-core launches
};

struct DionParams {
  DionMat mat[kChunk];
  int32_t n;    // matrices in this launch
  int32_t z0;   // group index of mat[0]
  DionDims d;
  DionBuf w;
};

// ---------------------------------------------------------------- stage: B = M + G

// Units of 8 columns over the zero-padded rows of Bw; blockIdx.y = matrix of the launch.
__global__ void __launch_bounds__(256) dion_stage_kernel(const __grid_constant__ DionParams p) {
  const DionMat& e = p.mat[blockIdx.y];
  const int z = p.z0 + int(blockIdx.y);
  const DionDims& d = p.d;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    OutEntry o;
    o.bits = nullptr;
    o.out = p.w.P0 + size_t(z) * d.m * d.ldr;
    o.ld = d.ldr;
    o.dtype = MAO_F32;
    o.flags = OUT_VEC;
    p.w.tP[z] = o;
    o.out = p.w.Rf + size_t(z) * d.n * d.ldr;
    p.w.tR[z] = o;
    o.out = e.M;
    o.ld = e.ldm;
    o.dtype = e.dtm;
    o.flags = e.flags_m;
    p.w.tM[z] = o;
    o.out = e.X;
    o.ld = e.ldx;
    o.dtype = e.dtx;
    o.flags = e.flags_x;
    p.w.tX[z] = o;
  }
  const int64_t upr = d.ldn / 8;
  const int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= d.m * upr) return;
  const int64_t row = u / upr, col0 = (u - row * upr) * 8;
  __nv_bfloat16* bw = p.w.Bw + (size_t(z) * d.m + row) * d.ldn + col0;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int64_t j = col0 + c;
    float b = 0.0f;
    if (j < d.n) {
      b = load_elem(e.M, row * e.ldm + j, e.dtm) + load_elem(e.G, row * e.ldg + j, e.dtg);
      store_elem(e.M, row * e.ldm + j, e.dtm, b);
      b = load_elem(e.M, row * e.ldm + j, e.dtm);  // B as stored (the update's residual)
    }
    bw[c] = __float2bfloat16_rn(b);
  }
}

// Qw = bf16(Q_prev), zero-padded to ldr columns.
__global__ void __launch_bounds__(256) dion_stage_q_kernel(const __grid_constant__ DionParams p) {
  const DionMat& e = p.mat[blockIdx.y];
  const int z = p.z0 + int(blockIdx.y);
  const DionDims& d = p.d;
  const int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= d.n * d.ldr) return;
  const int64_t i = u / d.ldr, j = u - i * d.ldr;
  p.w.Qw[(size_t(z) * d.n + i) * d.ldr + j] =
      __float2bfloat16_rn(j < d.r ? e.Q[i * e.ldq + j] : 0.0f);
}

// ------------------------------------------------------- Cholesky QR: S = P^T P

// Lower 64 x 64 tile (ti >= tj) of the partial Gram of rows [c*kGramRows, ...) of P;
// grid (tile pairs, row chunks, matrices). 256 threads, 4 x 4 outputs each.
__global__ void __launch_bounds__(256) dion_gram_kernel(const __grid_constant__ DionParams p,
                                                        const float* __restrict__ P) {
  const DionDims& d = p.d;
  const int z = p.z0 + int(blockIdx.z);
  int ti = 0, t = int(blockIdx.x);
  while (t > ti) { t -= ti + 1; ++ti; }
  const int tj = t;
  const int64_t r0 = int64_t(blockIdx.y) * kGramRows;
  const int64_t r1 = min(d.m, r0 + kGramRows);
  __shared__ float As[32][64 + 4], Bs[32][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  const float* Pz = P + size_t(z) * d.m * d.ldr;
  for (int64_t k0 = r0; k0 < r1; k0 += 32) {
    for (int q = threadIdx.x; q < 32 * 64; q += 256) {
      const int kk = q >> 6, c = q & 63;
      const int64_t row = k0 + kk;
      const int64_t ca = int64_t(ti) * 64 + c, cb = int64_t(tj) * 64 + c;
      As[kk][c] = (row < r1 && ca < d.r) ? Pz[row * d.ldr + ca] : 0.0f;
      Bs[kk][c] = (row < r1 && cb < d.r) ? Pz[row * d.ldr + cb] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        a[x] = As[kk][ty * 4 + x];
        b[x] = Bs[kk][tx * 4 + x];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = __fmaf_rn(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
  float* S = p.w.S + (size_t(z) * d.nchunks + blockIdx.y) * d.r * d.r;
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int64_t i = int64_t(ti) * 64 + ty * 4 + x, j = int64_t(tj) * 64 + tx * 4 + y;
      if (i < d.r && j < d.r) S[i * d.r + j] = acc[x][y];
    }
}

__device__ __forceinline__ int tri(int i, int j) { return i * (i + 1) / 2 + j; }  // j <= i

// One CTA per matrix: S (sum of the partial Grams, fixed order) = L L^T by right-looking
// Cholesky in shared memory (packed lower triangle), then Linv = L^-1 one column per warp
// by forward substitution. A pivot that is not positive sets the device error word and is
// replaced by 1e-30 (the caller's P had dependent columns).
__global__ void __launch_bounds__(1024) dion_chol_kernel(const __grid_constant__ DionParams p) {
  extern __shared__ float L[];  // r(r+1)/2 packed lower triangle, then 32 warps x r
  const DionDims& d = p.d;
  const int r = int(d.r);
  const int z = p.z0 + int(blockIdx.x);
  const float* S = p.w.S + size_t(z) * d.nchunks * r * r;
  const int ntri = r * (r + 1) / 2;
  for (int q = threadIdx.x; q < ntri; q += blockDim.x) {
    int i = int((sqrtf(8.0f * q + 1.0f) - 1.0f) * 0.5f);
    while (tri(i, 0) > q) --i;
    while (tri(i + 1, 0) <= q) ++i;
    const int j = q - tri(i, 0);
    float s = 0.0f;
    for (int c = 0; c < int(d.nchunks); ++c) s += S[size_t(c) * r * r + size_t(i) * r + j];
    L[q] = s;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int j = 0; j < r; ++j) {
    if (threadIdx.x == 0) {
      float piv = L[tri(j, j)];
      if (!(piv > 0.0f)) {
        atomicOr(&g_dion_error, 1u);
        piv = 1e-30f;
      }
      L[tri(j, j)] = sqrtf(piv);
    }
    __syncthreads();
    const float djj = L[tri(j, j)];
    for (int i = j + 1 + threadIdx.x; i < r; i += blockDim.x) L[tri(i, j)] /= djj;
    __syncthreads();
    for (int i = j + 1 + warp; i < r; i += nwarps) {
      const float lij = L[tri(i, j)];
      for (int k = j + 1 + lane; k <= i; k += 32) L[tri(i, k)] -= lij * L[tri(k, j)];
    }
    __syncthreads();
  }
  // Linv column c: x_c = 1 / L_cc, x_i = -(sum_{c<=k<i} L_ik x_k) / L_ii for i > c
  float* x = L + ntri + warp * r;
  float* Li = p.w.Linv + size_t(z) * r * r;
  for (int c = warp; c < r; c += nwarps) {
    for (int i = lane; i < r; i += 32) x[i] = 0.0f;
    __syncwarp();
    if (lane == 0) x[c] = 1.0f / L[tri(c, c)];
    __syncwarp();
    for (int i = c + 1; i < r; ++i) {
      float s = 0.0f;
      for (int k = c + lane; k < i; k += 32) s = __fmaf_rn(L[tri(i, k)], x[k], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
      if (lane == 0) x[i] = -s / L[tri(i, i)];
      __syncwarp();
    }
    for (int i = lane; i < r; i += 32) Li[size_t(i) * r + c] = x[i];
    __syncwarp();
  }
}

// Pout = Pin Linv^T (row i: x with x L^T = p), 64 x 64 output tiles, k only up to the
// tile's last column (Linv is lower triangular). The last pass also writes the bf16
// operand copy Pw (zero padding up to ldr) and the caller's optional P copy.
__global__ void __launch_bounds__(256) dion_trmul_kernel(const __grid_constant__ DionParams p,
                                                         const float* __restrict__ Pin,
                                                         float* __restrict__ Pout, int last) {
  const DionDims& d = p.d;
  const int z = p.z0 + int(blockIdx.z);
  const int64_t i0 = int64_t(blockIdx.x) * 64;
  const int j0 = int(blockIdx.y) * 64;
  const int r = int(d.r);
  __shared__ float As[32][64 + 4], Bs[32][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  const float* Pz = Pin + size_t(z) * d.m * d.ldr;
  const float* Li = p.w.Linv + size_t(z) * r * r;
  const int kend = min(r, j0 + 64);
  for (int k0 = 0; k0 < kend; k0 += 32) {
    for (int q = threadIdx.x; q < 32 * 64; q += 256) {
      const int kk = q >> 6, c = q & 63;
      const int k = k0 + kk;
      const int64_t row = i0 + c;
      const int col = j0 + c;
      As[kk][c] = (k < r && row < d.m) ? Pz[row * d.ldr + k] : 0.0f;
      Bs[kk][c] = (k < r && col < r) ? Li[size_t(col) * r + k] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        a[x] = As[kk][ty * 4 + x];
        b[x] = Bs[kk][tx * 4 + x];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = __fmaf_rn(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
  const DionMat& e = p.mat[blockIdx.z];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t i = i0 + ty * 4 + x;
    if (i >= d.m) continue;
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int j = j0 + tx * 4 + y;  // j < ldr (the grid covers ldr / 64 column tiles)
      const float v = j < r ? acc[x][y] : 0.0f;
      if (j < r) Pout[(size_t(z) * d.m + i) * d.ldr + j] = v;
      if (last) {
        p.w.Pw[(size_t(z) * d.m + i) * d.ldr + j] = __float2bfloat16_rn(v);
        if (e.Pout && j < r) e.Pout[i * r + j] = v;
      }
    }
  }
}

// ------------------------------------------------------ R -> Q = ColumnNormalize(R)

// Column norms of R (n x r): grid (ceil(r / 64), matrices); 4 row phases per column,
// summed in a fixed order.
__global__ void __launch_bounds__(256) dion_colnorm_kernel(const __grid_constant__ DionParams p) {
  const DionDims& d = p.d;
  const int z = p.z0 + int(blockIdx.y);
  const int c = threadIdx.x & 63, phase = threadIdx.x >> 6;
  const int64_t j = int64_t(blockIdx.x) * 64 + c;
  const float* R = p.w.Rf + size_t(z) * d.n * d.ldr;
  float s = 0.0f;
  if (j < d.r)
    for (int64_t i = phase; i < d.n; i += 4) {
      const float v = R[i * d.ldr + j];
      s = __fmaf_rn(v, v, s);
    }
  __shared__ float part[4][64];
  part[phase][c] = s;
  __syncthreads();
  if (phase == 0 && j < d.r)
    p.w.cn[size_t(z) * d.r + j] = sqrtf(((part[0][c] + part[1][c]) + part[2][c]) + part[3][c]);
}

// Q = R / c (a zero column stays zero) into the caller's Q, and the bf16 copies Qw, Rw.
__global__ void __launch_bounds__(256) dion_q_kernel(const __grid_constant__ DionParams p) {
  const DionMat& e = p.mat[blockIdx.y];
  const DionDims& d = p.d;
  const int z = p.z0 + int(blockIdx.y);
  const int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= d.n * d.ldr) return;
  const int64_t i = u / d.ldr, j = u - i * d.ldr;
  const size_t o = (size_t(z) * d.n + i) * d.ldr + j;
  float rv = 0.0f, qv = 0.0f;
  if (j < d.r) {
    rv = p.w.Rf[o];
    const float c = p.w.cn[size_t(z) * d.r + j];
    qv = c > 0.0f ? rv / c : 0.0f;
    e.Q[i * e.ldq + j] = qv;
  }
  p.w.Qw[o] = __float2bfloat16_rn(qv);
  p.w.Rw[o] = __float2bfloat16_rn(rv);
}

// ----------------------------------------------------------------- orchestration

struct DionLayout {
  DionDims d;
  size_t off_bw, off_qw, off_rw, off_pw, off_p0, off_p1, off_rf, off_s, off_linv, off_cn;
  size_t off_tables, total;
};

DionLayout dion_layout(int64_t m, int64_t n, int64_t r, int64_t count) {
  DionLayout L;
  L.d.m = m;
  L.d.n = n;
  L.d.r = r;
  L.d.ldn = round_up(n, tc::LD_ALIGN);
  L.d.ldr = round_up(r, tc::LD_ALIGN);
  L.d.nchunks = ceil_div(m, kGramRows);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = size_t(round_up(int64_t(off + bytes), 1024));
    return at;
  };
  const size_t c = size_t(count);
  L.off_bw = take(c * m * L.d.ldn * 2);
  L.off_qw = take(c * n * L.d.ldr * 2);
  L.off_rw = take(c * n * L.d.ldr * 2);
  L.off_pw = take(c * m * L.d.ldr * 2);
  L.off_p0 = take(c * m * L.d.ldr * 4);
  L.off_p1 = take(c * m * L.d.ldr * 4);
  L.off_rf = take(c * n * L.d.ldr * 4);
  L.off_s = take(c * L.d.nchunks * r * r * 4);
  L.off_linv = take(c * r * r * 4);
  L.off_cn = take(c * r * 4);
  L.off_tables = take(4 * c * sizeof(OutEntry));
  L.total = off;
  return L;
}

DionBuf dion_buffers(const DionLayout& L, uint8_t* ws, int64_t count) {
  DionBuf b;
  b.Bw = reinterpret_cast<__nv_bfloat16*>(ws + L.off_bw);
  b.Qw = reinterpret_cast<__nv_bfloat16*>(ws + L.off_qw);
  b.Rw = reinterpret_cast<__nv_bfloat16*>(ws + L.off_rw);
  b.Pw = reinterpret_cast<__nv_bfloat16*>(ws + L.off_pw);
  b.P0 = reinterpret_cast<float*>(ws + L.off_p0);
  b.P1 = reinterpret_cast<float*>(ws + L.off_p1);
  b.Rf = reinterpret_cast<float*>(ws + L.off_rf);
  b.S = reinterpret_cast<float*>(ws + L.off_s);
  b.Linv = reinterpret_cast<float*>(ws + L.off_linv);
  b.cn = reinterpret_cast<float*>(ws + L.off_cn);
  OutEntry* t = reinterpret_cast<OutEntry*>(ws + L.off_tables);
  b.tP = t;
  b.tR = t + count;
  b.tM = t + 2 * count;
  b.tX = t + 3 * count;
  return b;
}

// One tensor-core launch over the group: out-table product of A (rowsA x ldA) and B.
mao_status dion_tc(const void* srcA, int64_t rowsA, int64_t ldA, int a_mn, const void* srcB,
                   int64_t rowsB, int64_t ldB, int b_mn, int64_t M, int64_t N, int64_t K,
                   int64_t count, int stage, float alpha, const OutEntry* table,
                   cudaStream_t stream) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.ngroups = 1;
  p.stage = stage;
  p.a = alpha;
  p.scale = nullptr;
  p.out_table = table;
  p.timeout_ns = 4000000000ull;
  TcGroup& G = p.g[0];
  G.count = int32_t(count);
  G.slot0 = 0;
  G.a_mn = a_mn;
  G.b_mn = b_mn;
  G.M = int32_t(M);
  G.N = int32_t(N);
  G.K = int32_t(K);
  G.orig_cols = int32_t(N);
  G.final_out = 1;
  mao_status st = tc_encode_map(&G.tmA, srcA, rowsA, ldA, count);
  if (st == MAO_OK) st = tc_encode_map(&G.tmB, srcB, rowsB, ldB, count);
  if (st != MAO_OK) return st;
  G.tiles_m = int32_t(ceil_div(M, tc::TILE_M));
  G.tiles_n = int32_t(ceil_div(N, tc::BN));
  G.tiles_per_mat = G.tiles_m * G.tiles_n;
  G.tile_begin = 0;
  const int64_t tiles = int64_t(G.tiles_per_mat) * count;
  if (tiles > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
  p.total_tiles = int32_t(tiles);
  return tc_gemm_launch(p, stream);
}

int out_flags(const mao_mat& a) {
  return (reinterpret_cast<uintptr_t>(a.data) % 16 == 0 && (a.ld * elem_size(a.dtype)) % 16 == 0)
             ? OUT_VEC
             : 0;
}

}  // namespace

size_t dion_workspace_size(int64_t m, int64_t n, int64_t r, int64_t count) {
  return dion_layout(m, n, r, count).total;
}

mao_status dion_run(const mao_mat* X, const mao_mat* M, const mao_mat* G, const mao_mat* Q,
                    float* const* P_out, int32_t batch, int32_t rank, float mu, float lr,
                    void* workspace, cudaStream_t stream) {
  const int64_t m = X[0].rows, n = X[0].cols, r = rank;
  const DionLayout L = dion_layout(m, n, r, batch);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const DionBuf W = dion_buffers(L, ws, batch);
  const DionDims& d = L.d;
  static std::once_flag attr_once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  const size_t chol_smem = sizeof(float) * (size_t(r) * (r + 1) / 2 + 32 * size_t(r));
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(dion_chol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(sizeof(float) * (kMaxRank * (kMaxRank + 1) / 2 + 32 * kMaxRank)));
  });
  if (attr_err != cudaSuccess) return MAO_ERR_CUDA;

  // parameter blocks of up to kChunk matrices
  std::vector<DionParams> chunks;
  for (int z0 = 0; z0 < batch; z0 += kChunk) {
    DionParams p;
    memset(&p, 0, sizeof(p));
    p.n = std::min(kChunk, batch - z0);
    p.z0 = z0;
    p.d = d;
    p.w = W;
    for (int k = 0; k < p.n; ++k) {
      DionMat& e = p.mat[k];
      const int b = z0 + k;
      e.M = M[b].data;
      e.G = G[b].data;
      e.X = X[b].data;
      e.Q = reinterpret_cast<float*>(Q[b].data);
      e.Pout = P_out ? P_out[b] : nullptr;
      e.ldm = M[b].ld;
      e.ldg = G[b].ld;
      e.ldx = X[b].ld;
      e.ldq = Q[b].ld;
      e.dtm = M[b].dtype;
      e.dtg = G[b].dtype;
      e.dtx = X[b].dtype;
      e.flags_m = out_flags(M[b]);
      e.flags_x = out_flags(X[b]);
    }
    chunks.push_back(p);
  }
  auto grid = [](int64_t units, int y) { return dim3(unsigned(ceil_div(units, 256)), unsigned(y)); };
  auto check = [] {
    count_launch();
    return cudaGetLastError() == cudaSuccess;
  };
  // 1. B = M + G (M <- B), Bw; Qw = bf16(Q_prev); output tables
  for (const auto& p : chunks) {
    dion_stage_kernel<<<grid(d.m * (d.ldn / 8), p.n), 256, 0, stream>>>(p);
    if (!check()) return MAO_ERR_CUDA;
    dion_stage_q_kernel<<<grid(d.n * d.ldr, p.n), 256, 0, stream>>>(p);
    if (!check()) return MAO_ERR_CUDA;
  }
  // 2. P = B Q_prev (fp32)
  mao_status st = dion_tc(W.Bw, m, d.ldn, 0, W.Qw, n, d.ldr, 1, m, r, n, batch, NS_APPLY, 1.0f,
                          W.tP, stream);
  if (st != MAO_OK) return st;
  // 3. Cholesky QR, twice: P0 -> P1 -> P0 (+ Pw, caller's P)
  const int T = int(ceil_div(r, 64));
  for (int pass = 0; pass < 2; ++pass) {
    const float* Pin = pass == 0 ? W.P0 : W.P1;
    float* Pout = pass == 0 ? W.P1 : W.P0;
    for (const auto& p : chunks) {
      dion_gram_kernel<<<dim3(unsigned(T * (T + 1) / 2), unsigned(d.nchunks), unsigned(p.n)), 256, 0,
                         stream>>>(p, Pin);
      if (!check()) return MAO_ERR_CUDA;
      dion_chol_kernel<<<unsigned(p.n), 1024, chol_smem, stream>>>(p);
      if (!check()) return MAO_ERR_CUDA;
      dion_trmul_kernel<<<dim3(unsigned(ceil_div(m, 64)), unsigned(d.ldr / 64), unsigned(p.n)), 256,
                          0, stream>>>(p, Pin, Pout, pass == 1 ? 1 : 0);
      if (!check()) return MAO_ERR_CUDA;
    }
  }
  // 4. R = B^T P (fp32)
  st = dion_tc(W.Bw, m, d.ldn, 1, W.Pw, m, d.ldr, 1, n, r, m, batch, NS_APPLY, 1.0f, W.tR,
               stream);
  if (st != MAO_OK) return st;
  // 5. Q = ColumnNormalize(R) (caller's Q), bf16 copies of Q and R
  for (const auto& p : chunks) {
    dion_colnorm_kernel<<<dim3(unsigned(T), unsigned(p.n)), 256, 0, stream>>>(p);
    if (!check()) return MAO_ERR_CUDA;
    dion_q_kernel<<<grid(d.n * d.ldr, p.n), 256, 0, stream>>>(p);
    if (!check()) return MAO_ERR_CUDA;
  }
  // 6. M <- B - (1 - mu) P R^T ; X <- X - lr P Q^T (in place)
  st = dion_tc(W.Pw, m, d.ldr, 0, W.Rw, n, d.ldr, 0, m, n, r, batch, TC_UPDATE, -(1.0f - mu),
               W.tM, stream);
  if (st != MAO_OK) return st;
  return dion_tc(W.Pw, m, d.ldr, 0, W.Qw, n, d.ldr, 0, m, n, r, batch, TC_UPDATE, -lr, W.tX,
                 stream);
}

mao_status dion_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_dion_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MAO_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MAO_ERR_CUDA;
  if (v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_dion_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
      return MAO_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MAO_ERR_CUDA;
    return MAO_ERR_NUMERIC;
  }
  return MAO_OK;
}

}  // namespace mao

using namespace mao;

extern "C" {

size_t dion_workspace_bytes(const mao_mat* X, int32_t batch, int32_t rank) {
  if (!X || batch < 1 || rank < 1 || rank > kMaxRank) return 0;
  if (X[0].rows < 1 || X[0].cols < 1 || X[0].rows > (int64_t(1) << 31) ||
      X[0].cols > (int64_t(1) << 31))
    return 0;
  if (rank > std::min(X[0].rows, X[0].cols)) return 0;
  return dion_workspace_size(X[0].rows, X[0].cols, rank, batch);
}

mao_status dion_step(const mao_mat* X, const mao_mat* M, const mao_mat* G, const mao_mat* Q,
                     float* const* P_out, int32_t batch, int32_t rank, float mu, float lr,
                     int32_t compute, void* workspace, size_t workspace_bytes, void* stream) {
  if (!X || !M || !G || !Q || batch < 1 || rank < 1 || rank > kMaxRank) return MAO_ERR_INVALID_ARG;
  if (!std::isfinite(mu) || !std::isfinite(lr)) return MAO_ERR_INVALID_ARG;
  if (compute != MAO_BF16) return MAO_ERR_UNSUPPORTED;
  const int64_t m = X[0].rows, n = X[0].cols;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_mat(X[b]);
    if (st == MAO_OK) st = check_mat(M[b]);
    if (st == MAO_OK) st = check_mat(G[b]);
    if (st == MAO_OK) st = check_mat(Q[b]);
    if (st != MAO_OK) return st;
    if (X[b].rows != m || X[b].cols != n || M[b].rows != m || M[b].cols != n ||
        G[b].rows != m || G[b].cols != n)
      return MAO_ERR_INVALID_ARG;
    if (Q[b].dtype != MAO_F32 || Q[b].rows != n || Q[b].cols != rank) return MAO_ERR_INVALID_ARG;
    if (P_out && P_out[b] && reinterpret_cast<uintptr_t>(P_out[b]) % 4 != 0)
      return MAO_ERR_MISALIGNED;
  }
  if (rank > std::min(m, n)) return MAO_ERR_INVALID_ARG;
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < dion_workspace_size(m, n, rank, batch)) return MAO_ERR_WORKSPACE;
  return dion_run(X, M, G, Q, P_out, batch, rank, mu, lr, workspace,
                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
