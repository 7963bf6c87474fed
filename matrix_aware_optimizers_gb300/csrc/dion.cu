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
// diagonal, computed as Cholesky QR applied twice: S = P^T P, S = L L^T, P <- P L^-T
// (a blocked forward substitution with the inverses of L's 32 x 32 diagonal blocks).
// The three dense products run on the same tcgen05 kernel as Newton–Schulz, over up to
// eight shape groups per launch; the r x r work (Gram matrices, Cholesky, triangular
// solve) runs in fp32 on CUDA cores, every matrix of the call in one launch per stage.
// Per-matrix descriptors live in a device table in the workspace (written by a set-up
// kernel), so a call of any size and any mix of shapes takes a fixed number of launches.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "ns_plan.h"

namespace mao {

__device__ unsigned int g_dion_error;  // bit 0: a Cholesky pivot was not positive

namespace {

constexpr int kMaxRank = 256;
constexpr int kGramRows = 1024;   // rows of P summed by one partial Gram tile
constexpr int kNormRows = 256;    // rows of R summed by one partial column norm
constexpr int kSetup = 16;        // table entries written per set-up launch
constexpr int kCholThreads = 512;

// Everything the CUDA-core kernels need about one matrix slot.
struct DionSlot {
  void* M;
  const void* G;
  void* X;
  float* Q;
  float* Pout;                      // optional copy of the final P (m x r, row stride r)
  __nv_bfloat16 *Bw, *Qw, *Rw, *Pw; // bf16 operands, rows of ldn / ldr elements
  float *P0, *P1, *Rf;              // fp32 [m|n][ldr]
  float *S, *L, *D, *cn;            // [gchunks][r][r]; L [r][r]; [nb][32][32]; [nchunks + 1][r]
  int64_t ldm, ldg, ldx, ldq;
  int32_t m, n, ldn;
  int32_t dtm, dtg, dtx;
  int32_t flags_m, flags_x;
  int32_t gchunks, nchunks;         // partial Gram row chunks of P, partial norm chunks of R
  int32_t vec;                      // M and G: bf16/f32 rows that allow 16-byte accesses
};

struct DionCommon {
  const DionSlot* slots;            // device table [count]
  OutEntry *tP, *tR, *tM, *tX;      // output tables of the tensor-core launches [count]
  int32_t r, ldr, count;
};

struct SetupParams {
  DionSlot s[kSetup];
  int32_t n, z0;
  DionCommon c;
};

// ---------------------------------------------------------------- set-up

// Thread k writes slot z0 + k of the device table and its four output entries.
__global__ void dion_setup_kernel(const __grid_constant__ SetupParams p) {
  const int k = threadIdx.x;
  if (k >= p.n) return;
  const DionSlot& e = p.s[k];
  const int z = p.z0 + k;
  const_cast<DionSlot*>(p.c.slots)[z] = e;
  OutEntry o;
  o.bits = nullptr;
  o.out = e.P0;
  o.ld = p.c.ldr;
  o.dtype = MAO_F32;
  o.flags = OUT_VEC;
  p.c.tP[z] = o;
  o.out = e.Rf;
  p.c.tR[z] = o;
  o.out = e.M;
  o.ld = e.ldm;
  o.dtype = e.dtm;
  o.flags = e.flags_m;
  p.c.tM[z] = o;
  o.out = e.X;
  o.ld = e.ldx;
  o.dtype = e.dtx;
  o.flags = e.flags_x;
  p.c.tX[z] = o;
}

// ---------------------------------------------------------------- B = M + G, Qw

__device__ __forceinline__ float round_to(float v, int32_t dt) {
  return dt == MAO_BF16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// Units of 8 columns over the zero-padded rows of Bw; blockIdx.y = slot. M <- M + G in
// place (rounded to M's dtype) and Bw = bf16 of the stored B.
__global__ void __launch_bounds__(256) dion_stage_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.y];
  const uint32_t upr = uint32_t(e.ldn) / 8;
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= uint32_t(e.m) * upr) return;
  const int64_t row = u / upr, col0 = int64_t(u - uint32_t(row) * upr) * 8;
  float b[8];
  if (e.vec && col0 + 8 <= e.n) {
    float mv[8], gv[8];
    load8(e.M, row * e.ldm + col0, e.dtm, mv);
    load8(e.G, row * e.ldg + col0, e.dtg, gv);
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = mv[k] + gv[k];
    store8(e.M, row * e.ldm + col0, e.dtm, b);
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = round_to(b[k], e.dtm);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t j = col0 + k;
      b[k] = 0.0f;
      if (j < e.n) {
        const float v = load_elem(e.M, row * e.ldm + j, e.dtm) + load_elem(e.G, row * e.ldg + j, e.dtg);
        store_elem(e.M, row * e.ldm + j, e.dtm, v);
        b[k] = round_to(v, e.dtm);
      }
    }
  }
  store8(e.Bw, row * e.ldn + col0, MAO_BF16, b);
}

// Qw = bf16(Q_prev), zero-padded to ldr columns; blockIdx.y = slot.
__global__ void __launch_bounds__(256) dion_stage_q_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.y];
  const uint32_t upr = uint32_t(c.ldr) / 8;
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= uint32_t(e.n) * upr) return;
  const uint32_t i = u / upr, j0 = (u - i * upr) * 8;
  float v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int j = int(j0) + k;
    v[k] = j < c.r ? e.Q[size_t(i) * e.ldq + j] : 0.0f;
  }
  store8(e.Qw, size_t(i) * c.ldr + j0, MAO_BF16, v);
}

// ------------------------------------------------------- Cholesky QR: S = P^T P

// Lower 64 x 64 tile (ti >= tj) of the partial Gram of rows [chunk*kGramRows, ...) of P;
// grid (tile pairs, row chunks, slots). 256 threads, 4 x 4 outputs each.
__global__ void __launch_bounds__(256) dion_gram_kernel(const __grid_constant__ DionCommon c,
                                                        int from_p1) {
  const DionSlot& e = c.slots[blockIdx.z];
  if (int(blockIdx.y) >= e.gchunks) return;
  int ti = 0, t = int(blockIdx.x);
  while (t > ti) { t -= ti + 1; ++ti; }
  const int tj = t;
  const int r = c.r;
  const int64_t r0 = int64_t(blockIdx.y) * kGramRows;
  const int64_t r1 = min(int64_t(e.m), r0 + kGramRows);
  __shared__ float As[32][64 + 4], Bs[32][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  const float* P = from_p1 ? e.P1 : e.P0;
  for (int64_t k0 = r0; k0 < r1; k0 += 32) {
    for (int q = threadIdx.x; q < 32 * 64; q += 256) {
      const int kk = q >> 6, cc = q & 63;
      const int64_t row = k0 + kk;
      const int ca = ti * 64 + cc, cb = tj * 64 + cc;
      As[kk][cc] = (row < r1 && ca < r) ? P[row * c.ldr + ca] : 0.0f;
      Bs[kk][cc] = (row < r1 && cb < r) ? P[row * c.ldr + cb] : 0.0f;
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
  float* S = e.S + size_t(blockIdx.y) * r * r;
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int i = ti * 64 + ty * 4 + x, j = tj * 64 + tx * 4 + y;
      if (i < r && j < r) S[size_t(i) * r + j] = acc[x][y];
    }
}

// Lower blocks of a matrix cut into 32 x 32 blocks, block (I, J) with I >= J at index
// I (I + 1) / 2 + J, each block 32 rows of 33 floats (the pad keeps column reads of a warp
// on distinct banks).
__device__ __forceinline__ float* blk(float* A, int I, int J) {
  return A + (I * (I + 1) / 2 + J) * (32 * 33);
}

// One CTA per slot: S (the partial Grams added in chunk order) = L L^T by blocked
// right-looking Cholesky with 32 x 32 blocks in shared memory. For each block column J:
//   warp 0 factors the diagonal block (unscaled right-looking steps, then column scaling)
//   and inverts it (D_J, lane = column, forward substitution in registers);
//   the panel below is L_IJ = A_IJ D_J^T (one warp per row, lane = column);
//   every trailing lower block gets A_IK -= L_IJ L_KJ^T (one warp per block, lane =
//   column, the lane's row of L_KJ held in registers).
// A pivot that is not positive sets the device error word and is replaced by 1e-30 (P had
// dependent columns). Rows and columns past r are the identity. L goes to global memory
// (row-major, zeros above the diagonal) and D_J to e.D.
__global__ void __launch_bounds__(kCholThreads, 1) dion_chol_kernel(const __grid_constant__ DionCommon c) {
  extern __shared__ float sm[];
  const DionSlot& e = c.slots[blockIdx.x];
  const int r = c.r;
  const int nb = (r + 31) / 32;
  float* A = sm;                                // nb (nb + 1) / 2 blocks
  float* Dsm = sm + nb * (nb + 1) / 2 * 32 * 33;  // [32][33], the current D_J
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int kWarps = kCholThreads / 32;
  const int gch = e.gchunks;
  const float* S = e.S;
  // load the lower blocks (rows i >= k in the diagonal blocks), identity past r
  for (int b = warp; b < nb * (nb + 1) / 2; b += kWarps) {
    int I = 0, J = b;
    while (J > I) { J -= I + 1; ++I; }
    float* Ab = blk(A, I, J);
    for (int ii = 0; ii < 32; ++ii) {
      const int i = 32 * I + ii, k = 32 * J + lane;
      float v = 0.0f;
      if (i < r && k < r && k <= i)
        for (int ch = 0; ch < gch; ++ch) v += S[(size_t(ch) * r + i) * r + k];
      else if (i == k)
        v = 1.0f;
      Ab[ii * 33 + lane] = v;
    }
  }
  __syncthreads();
  for (int J = 0; J < nb; ++J) {
    if (warp == 0) {
      float* Ad = blk(A, J, J);
      // right-looking steps on unscaled columns: at step j, lane k > j updates its column k
      // below the diagonal, A_ik -= A_ij A_kj / A_jj for i >= k (column j is only read)
      for (int j = 0; j < 32; ++j) {
        float pj = Ad[j * 33 + j];
        if (!(pj > 0.0f)) {
          if (lane == 0) atomicOr(&g_dion_error, 1u);
          pj = 1e-30f;
        }
        if (lane > j) {
          const float akj = Ad[lane * 33 + j] / pj;
          for (int i = lane; i < 32; ++i) Ad[i * 33 + lane] = __fmaf_rn(-Ad[i * 33 + j], akj, Ad[i * 33 + lane]);
        }
        __syncwarp();
        if (lane == j) Ad[j * 33 + j] = pj;  // the sanitised pivot, kept for the scaling
        __syncwarp();
      }
      // L_ik = A_ik / sqrt(pivot_k) for k < i (lane = row), then L_ii = sqrt(pivot_i)
      for (int k = 0; k < lane; ++k) Ad[lane * 33 + k] *= rsqrtf(Ad[k * 33 + k]);
      __syncwarp();
      Ad[lane * 33 + lane] = sqrtf(Ad[lane * 33 + lane]);
      __syncwarp();
      // D_J = L_JJ^-1, lane = column
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < i; ++k) sum = __fmaf_rn(Ad[i * 33 + k], k >= lane ? x[k] : 0.0f, sum);
        const float lii = Ad[i * 33 + i];
        x[i] = i < lane ? 0.0f : (i == lane ? 1.0f / lii : -sum / lii);
      }
      float* D = e.D + size_t(J) * 32 * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        Dsm[i * 33 + lane] = x[i];
        D[i * 32 + lane] = x[i];
      }
    }
    __syncthreads();
    // panel: L_IJ = A_IJ D^T, one warp per row of the blocks below
    for (int row = 32 * (J + 1) + warp; row < 32 * nb; row += kWarps) {
      float* Ap = blk(A, row / 32, J) + (row % 32) * 33;
      float acc = 0.0f;
      for (int q = 0; q <= lane; ++q) acc = __fmaf_rn(Ap[q], Dsm[lane * 33 + q], acc);
      __syncwarp();
      Ap[lane] = acc;
    }
    __syncthreads();
    // trailing lower blocks (I, K), J < K <= I: one warp per block
    const int t = nb - J - 1;
    for (int b = warp; b < t * (t + 1) / 2; b += kWarps) {
      int I = 0, K = b;
      while (K > I) { K -= I + 1; ++I; }
      I += J + 1;
      K += J + 1;
      float lk[32];
      const float* Lk = blk(A, K, J) + lane * 33;
#pragma unroll
      for (int q = 0; q < 32; ++q) lk[q] = Lk[q];
      const float* Li = blk(A, I, J);
      float* Ab = blk(A, I, K);
      for (int ii = 0; ii < 32; ++ii) {
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 32; ++q) sum = __fmaf_rn(Li[ii * 33 + q], lk[q], sum);
        Ab[ii * 33 + lane] -= sum;
      }
    }
    __syncthreads();
  }
  // L to global memory, row-major r x r, zeros above the diagonal
  for (int q = threadIdx.x; q < r * r; q += kCholThreads) {
    const int i = q / r, k = q - i * r;
    e.L[q] = k <= i ? blk(A, i / 32, k / 32)[(i % 32) * 33 + (k % 32)] : 0.0f;
  }
}

// Pout = Pin L^-T by blocked forward substitution over 32-column blocks J:
//   Pout[:, J] = (Pin[:, J] - Pout[:, <J] L[J, <J]^T) D_J^T,   D_J = L[J, J]^-1.
// One CTA (256 threads, 8 rows x 1 column each) per 64 rows of one slot; the rows of Pout
// stay in shared memory, and the rows of L[J, <J] and D_J are staged there per block
// (coalesced loads). The last pass also writes the bf16 operand copy Pw (zero padding up
// to ldr) and the caller's P copy.
constexpr int kTrsmThreads = 256;

__global__ void __launch_bounds__(kTrsmThreads) dion_trsm_kernel(const __grid_constant__ DionCommon c,
                                                                 int pass) {
  extern __shared__ float tsm[];
  const DionSlot& e = c.slots[blockIdx.y];
  const int64_t i0 = int64_t(blockIdx.x) * 64;
  if (i0 >= e.m) return;
  const int r = c.r, ldr = c.ldr;
  const int pld = r + 1;
  float* Pn = tsm;              // [64][r + 1]
  float* T = Pn + 64 * pld;     // [64][33]
  float* Ls = T + 64 * 33;      // [32][r + 1]: rows of L[J, <J]
  float* Ds = Ls + 32 * pld;    // [32][33]: D_J
  const float* Pin = pass == 0 ? e.P0 : e.P1;
  float* Pout = pass == 0 ? e.P1 : e.P0;
  const int cc = threadIdx.x % 32, rg = threadIdx.x / 32;  // column in the block, row group
  const int nb = (r + 31) / 32;
  for (int J = 0; J < nb; ++J) {
    const int j0 = 32 * J;
    for (int q = threadIdx.x; q < 32 * j0; q += kTrsmThreads) {
      const int rr = q / j0, k = q - rr * j0;
      Ls[rr * pld + k] = (j0 + rr < r) ? e.L[size_t(j0 + rr) * r + k] : 0.0f;
    }
    for (int q = threadIdx.x; q < 32 * 32; q += kTrsmThreads)
      Ds[(q / 32) * 33 + q % 32] = e.D[size_t(J) * 1024 + q];
    const int gj = j0 + cc;
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int64_t row = i0 + rg * 8 + t;
      acc[t] = (row < e.m && gj < r) ? Pin[row * ldr + gj] : 0.0f;
    }
    __syncthreads();
    for (int k = 0; k < j0; ++k) {
      const float l = Ls[cc * pld + k];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = __fmaf_rn(-Pn[(rg * 8 + t) * pld + k], l, acc[t]);
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) T[(rg * 8 + t) * 33 + cc] = acc[t];
    __syncthreads();
    float out[8] = {};
    for (int q = 0; q <= cc; ++q) {
      const float d = Ds[cc * 33 + q];
#pragma unroll
      for (int t = 0; t < 8; ++t) out[t] = __fmaf_rn(T[(rg * 8 + t) * 33 + q], d, out[t]);
    }
    if (gj < r) {
#pragma unroll
      for (int t = 0; t < 8; ++t) Pn[(rg * 8 + t) * pld + gj] = out[t];
    }
    __syncthreads();
  }
  // write back: fp32 P (columns < r), bf16 Pw (columns < ldr), the caller's copy
  for (int q = threadIdx.x; q < 64 * ldr; q += kTrsmThreads) {
    const int t = q / ldr, j = q - t * ldr;
    const int64_t row = i0 + t;
    if (row >= e.m) continue;
    const float v = j < r ? Pn[t * pld + j] : 0.0f;
    if (j < r) Pout[row * ldr + j] = v;
    if (pass == 1) {
      e.Pw[row * ldr + j] = __float2bfloat16_rn(v);
      if (e.Pout && j < r) e.Pout[row * r + j] = v;
    }
  }
}

// ------------------------------------------------------ R -> Q = ColumnNormalize(R)

// Partial column sums of squares of R over rows [chunk*kNormRows, ...); grid
// (ceil(r / 64), row chunks, slots); 4 row phases per column, summed in a fixed order.
__global__ void __launch_bounds__(256) dion_colnorm_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.z];
  if (int(blockIdx.y) >= e.nchunks) return;
  const int cc = threadIdx.x & 63, phase = threadIdx.x >> 6;
  const int j = int(blockIdx.x) * 64 + cc;
  const int64_t r0 = int64_t(blockIdx.y) * kNormRows;
  const int64_t r1 = min(int64_t(e.n), r0 + kNormRows);
  float s = 0.0f;
  if (j < c.r)
    for (int64_t i = r0 + phase; i < r1; i += 4) {
      const float v = e.Rf[i * c.ldr + j];
      s = __fmaf_rn(v, v, s);
    }
  __shared__ float part[4][64];
  part[phase][cc] = s;
  __syncthreads();
  if (phase == 0 && j < c.r)
    e.cn[size_t(blockIdx.y) * c.r + j] = ((part[0][cc] + part[1][cc]) + part[2][cc]) + part[3][cc];
}

// Column norms: the partial sums added in chunk order, square root; one block per slot.
// The norms go after the partials (e.cn + nchunks * r).
__global__ void __launch_bounds__(256) dion_norm_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.x];
  for (int j = threadIdx.x; j < c.r; j += blockDim.x) {
    float ss = 0.0f;
    for (int ch = 0; ch < e.nchunks; ++ch) ss += e.cn[size_t(ch) * c.r + j];
    e.cn[size_t(e.nchunks) * c.r + j] = sqrtf(ss);
  }
}

// Q = R / c (a zero column stays zero) into the caller's Q, and the bf16 copies Qw, Rw;
// 8 columns per thread.
__global__ void __launch_bounds__(256) dion_q_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.y];
  const uint32_t upr = uint32_t(c.ldr) / 8;
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= uint32_t(e.n) * upr) return;
  const uint32_t i = u / upr, j0 = (u - i * upr) * 8;
  const float* cn = e.cn + size_t(e.nchunks) * c.r;
  float rv[8], qv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int j = int(j0) + k;
    rv[k] = 0.0f;
    qv[k] = 0.0f;
    if (j < c.r) {
      rv[k] = e.Rf[size_t(i) * c.ldr + j];
      const float nrm = cn[j];
      qv[k] = nrm > 0.0f ? rv[k] / nrm : 0.0f;
      e.Q[size_t(i) * e.ldq + j] = qv[k];
    }
  }
  store8(e.Qw, size_t(i) * c.ldr + j0, MAO_BF16, qv);
  store8(e.Rw, size_t(i) * c.ldr + j0, MAO_BF16, rv);
}

// ----------------------------------------------------------------- orchestration

struct DionGroup {
  int64_t m, n;
  int32_t count, slot0;
  size_t off_bw, off_qw, off_rw, off_pw, off_p0, off_p1, off_rf, off_s, off_l, off_d, off_cn;
};

struct DionPlan {
  std::vector<DionGroup> groups;
  std::vector<int> input_of;  // slot -> caller's index
  int64_t r = 0, ldr = 0;
  size_t off_slots = 0, off_tables = 0, total = 0;
  int64_t max_units = 0, max_qunits = 0, max_rowtiles = 0, max_gchunks = 0, max_nchunks = 0;
};

void make_dion_plan(const mao_mat* X, int32_t batch, int32_t rank, DionPlan& plan) {
  plan = DionPlan();
  plan.r = rank;
  plan.ldr = round_up(rank, tc::LD_ALIGN);
  std::map<std::pair<int64_t, int64_t>, int> gid;
  std::vector<std::vector<int>> members;
  for (int b = 0; b < batch; ++b) {
    const auto key = std::make_pair(X[b].rows, X[b].cols);
    auto it = gid.find(key);
    if (it == gid.end()) {
      gid.emplace(key, int(members.size()));
      members.push_back({b});
    } else {
      members[it->second].push_back(b);
    }
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = size_t(round_up(int64_t(off + bytes), 1024));
    return at;
  };
  plan.off_slots = take(sizeof(DionSlot) * size_t(batch));
  plan.off_tables = take(4 * sizeof(OutEntry) * size_t(batch));
  const size_t r = size_t(rank), ldr = size_t(plan.ldr);
  int slot = 0;
  for (const auto& mem : members) {
    DionGroup g;
    g.m = X[mem[0]].rows;
    g.n = X[mem[0]].cols;
    g.count = int32_t(mem.size());
    g.slot0 = slot;
    const size_t c = size_t(g.count), m = size_t(g.m), n = size_t(g.n);
    const size_t ldn = size_t(round_up(g.n, tc::LD_ALIGN));
    const size_t gch = size_t(ceil_div(g.m, kGramRows)), nch = size_t(ceil_div(g.n, kNormRows));
    g.off_bw = take(c * m * ldn * 2);
    g.off_qw = take(c * n * ldr * 2);
    g.off_rw = take(c * n * ldr * 2);
    g.off_pw = take(c * m * ldr * 2);
    g.off_p0 = take(c * m * ldr * 4);
    g.off_p1 = take(c * m * ldr * 4);
    g.off_rf = take(c * n * ldr * 4);
    g.off_s = take(c * gch * r * r * 4);
    g.off_l = take(c * r * r * 4);
    g.off_d = take(c * size_t(ceil_div(rank, 32)) * 32 * 32 * 4);
    g.off_cn = take(c * (nch + 1) * r * 4);
    for (int b : mem) plan.input_of.push_back(b);
    slot += g.count;
    plan.max_units = std::max<int64_t>(plan.max_units, g.m * int64_t(ldn / 8));
    plan.max_qunits = std::max<int64_t>(plan.max_qunits, g.n * int64_t(ldr / 8));
    plan.max_rowtiles = std::max<int64_t>(plan.max_rowtiles, ceil_div(g.m, 64));
    plan.max_gchunks = std::max<int64_t>(plan.max_gchunks, int64_t(gch));
    plan.max_nchunks = std::max<int64_t>(plan.max_nchunks, int64_t(nch));
    plan.groups.push_back(g);
  }
  plan.total = off;
}

int out_flags(const mao_mat& a) {
  return (reinterpret_cast<uintptr_t>(a.data) % 16 == 0 && (a.ld * elem_size(a.dtype)) % 16 == 0)
             ? OUT_VEC
             : 0;
}

// Tensor-core launches of one product over every group (up to eight groups per launch).
// op: 0 = P = B Q, 1 = R = B^T P, 2 = M update (P R^T), 3 = X update (P Q^T).
mao_status dion_tc(const DionPlan& plan, uint8_t* ws, const OutEntry* table, int op, float alpha,
                   cudaStream_t stream) {
  const int64_t r = plan.r, ldr = plan.ldr;
  for (size_t g0 = 0; g0 < plan.groups.size(); g0 += tc::MAX_GROUPS) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.stage = op >= 2 ? TC_UPDATE : NS_APPLY;
    p.a = alpha;
    p.scale = nullptr;
    p.out_table = table;
    p.timeout_ns = wait_limit_ns();
    int64_t tiles = 0;
    for (size_t gi = g0; gi < plan.groups.size() && p.ngroups < tc::MAX_GROUPS; ++gi) {
      const DionGroup& g = plan.groups[gi];
      TcGroup& G = p.g[p.ngroups++];
      const int64_t ldn = round_up(g.n, tc::LD_ALIGN);
      const void *A, *B;
      int64_t rowsA, ldA, rowsB, ldB;
      switch (op) {
        case 0:  // (m x n)(n x r): Bw K-major, Qw MN-major
          A = ws + g.off_bw; rowsA = g.m; ldA = ldn; G.a_mn = 0;
          B = ws + g.off_qw; rowsB = g.n; ldB = ldr; G.b_mn = 1;
          G.M = int32_t(g.m); G.N = int32_t(r); G.K = int32_t(g.n);
          break;
        case 1:  // (n x m)(m x r): Bw MN-major, Pw MN-major
          A = ws + g.off_bw; rowsA = g.m; ldA = ldn; G.a_mn = 1;
          B = ws + g.off_pw; rowsB = g.m; ldB = ldr; G.b_mn = 1;
          G.M = int32_t(g.n); G.N = int32_t(r); G.K = int32_t(g.m);
          break;
        default:  // (m x r)(r x n): Pw K-major, Rw / Qw K-major
          A = ws + g.off_pw; rowsA = g.m; ldA = ldr; G.a_mn = 0;
          B = ws + (op == 2 ? g.off_rw : g.off_qw); rowsB = g.n; ldB = ldr; G.b_mn = 0;
          G.M = int32_t(g.m); G.N = int32_t(g.n); G.K = int32_t(r);
          break;
      }
      G.count = g.count;
      G.slot0 = g.slot0;
      G.orig_cols = G.N;
      G.final_out = 1;
      mao_status st = tc_encode_map(&G.tmA, A, rowsA, ldA, g.count);
      if (st == MAO_OK) st = tc_encode_map(&G.tmB, B, rowsB, ldB, g.count);
      if (st != MAO_OK) return st;
      G.tiles_m = int32_t(ceil_div(G.M, tc::TILE_M));
      G.tiles_n = int32_t(ceil_div(G.N, tc::BN));
      G.tiles_per_mat = G.tiles_m * G.tiles_n;
      G.tile_begin = int32_t(tiles);
      tiles += int64_t(G.tiles_per_mat) * g.count;
      if (tiles > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
    }
    p.total_tiles = int32_t(tiles);
    const mao_status st = tc_gemm_launch(p, stream);
    if (st != MAO_OK) return st;
  }
  return MAO_OK;
}

}  // namespace

size_t dion_workspace_size(const mao_mat* X, int32_t batch, int32_t rank) {
  DionPlan plan;
  make_dion_plan(X, batch, rank, plan);
  return plan.total;
}

mao_status dion_run(const mao_mat* X, const mao_mat* M, const mao_mat* G, const mao_mat* Q,
                    float* const* P_out, int32_t batch, int32_t rank, float mu, float lr,
                    void* workspace, cudaStream_t stream) {
  DionPlan plan;
  make_dion_plan(X, batch, rank, plan);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  DionCommon c;
  c.slots = reinterpret_cast<const DionSlot*>(ws + plan.off_slots);
  OutEntry* tables = reinterpret_cast<OutEntry*>(ws + plan.off_tables);
  c.tP = tables;
  c.tR = tables + batch;
  c.tM = tables + 2 * batch;
  c.tX = tables + 3 * batch;
  c.r = rank;
  c.ldr = int32_t(plan.ldr);
  c.count = batch;

  static std::once_flag attr_once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  cudaError_t attr_err = cudaSuccess;
  auto chol_bytes = [](int rk) {
    const size_t nbk = size_t(ceil_div(rk, 32));
    return sizeof(float) * (nbk * (nbk + 1) / 2 * 32 * 33 + 32 * 33);
  };
  auto trsm_bytes = [](int rk) {
    return sizeof(float) * (96 * size_t(rk + 1) + 64 * 33 + 32 * 33);
  };
  const size_t chol_max = chol_bytes(kMaxRank), trsm_max = trsm_bytes(kMaxRank);
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(dion_chol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(chol_max));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(dion_trsm_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(trsm_max));
  });
  if (attr_err != cudaSuccess) return MAO_ERR_CUDA;
  auto launched = [] {
    count_launch();
    return cudaGetLastError() == cudaSuccess;
  };

  // 0. the device table of slots and the output tables
  std::vector<DionSlot> slots(batch);
  for (const auto& g : plan.groups) {
    const int64_t ldn = round_up(g.n, tc::LD_ALIGN);
    for (int k = 0; k < g.count; ++k) {
      const int z = g.slot0 + k;
      const int b = plan.input_of[z];
      DionSlot& e = slots[z];
      memset(&e, 0, sizeof(e));
      e.M = M[b].data;
      e.G = G[b].data;
      e.X = X[b].data;
      e.Q = reinterpret_cast<float*>(Q[b].data);
      e.Pout = P_out ? P_out[b] : nullptr;
      e.Bw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_bw) + size_t(k) * g.m * ldn;
      e.Qw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_qw) + size_t(k) * g.n * plan.ldr;
      e.Rw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_rw) + size_t(k) * g.n * plan.ldr;
      e.Pw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_pw) + size_t(k) * g.m * plan.ldr;
      e.P0 = reinterpret_cast<float*>(ws + g.off_p0) + size_t(k) * g.m * plan.ldr;
      e.P1 = reinterpret_cast<float*>(ws + g.off_p1) + size_t(k) * g.m * plan.ldr;
      e.Rf = reinterpret_cast<float*>(ws + g.off_rf) + size_t(k) * g.n * plan.ldr;
      e.gchunks = int32_t(ceil_div(g.m, kGramRows));
      e.nchunks = int32_t(ceil_div(g.n, kNormRows));
      e.S = reinterpret_cast<float*>(ws + g.off_s) + size_t(k) * e.gchunks * rank * rank;
      e.L = reinterpret_cast<float*>(ws + g.off_l) + size_t(k) * rank * rank;
      e.D = reinterpret_cast<float*>(ws + g.off_d) + size_t(k) * ceil_div(rank, 32) * 32 * 32;
      e.cn = reinterpret_cast<float*>(ws + g.off_cn) + size_t(k) * (e.nchunks + 1) * rank;
      e.ldm = M[b].ld;
      e.ldg = G[b].ld;
      e.ldx = X[b].ld;
      e.ldq = Q[b].ld;
      e.m = int32_t(g.m);
      e.n = int32_t(g.n);
      e.ldn = int32_t(ldn);
      e.dtm = M[b].dtype;
      e.dtg = G[b].dtype;
      e.dtx = X[b].dtype;
      e.flags_m = out_flags(M[b]);
      e.flags_x = out_flags(X[b]);
      e.vec = vec8_ok(M[b]) && vec8_ok(G[b]) ? 1 : 0;
    }
  }
  for (int z0 = 0; z0 < batch; z0 += kSetup) {
    SetupParams sp;
    memset(&sp, 0, sizeof(sp));
    sp.n = std::min(kSetup, batch - z0);
    sp.z0 = z0;
    sp.c = c;
    for (int k = 0; k < sp.n; ++k) sp.s[k] = slots[z0 + k];
    dion_setup_kernel<<<1, kSetup, 0, stream>>>(sp);
    if (!launched()) return MAO_ERR_CUDA;
  }
  const unsigned nb = unsigned(batch);
  auto blocks = [](int64_t units) { return unsigned(ceil_div(units, 256)); };
  // 1. B = M + G (M <- B), Bw; Qw = bf16(Q_prev)
  dion_stage_kernel<<<dim3(blocks(plan.max_units), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  dion_stage_q_kernel<<<dim3(blocks(plan.max_qunits), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  // 2. P = B Q_prev (fp32)
  mao_status st = dion_tc(plan, ws, c.tP, 0, 1.0f, stream);
  if (st != MAO_OK) return st;
  // 3. Cholesky QR, twice: P0 -> P1 -> P0 (+ Pw, caller's P)
  const int T = int(ceil_div(rank, 64));
  const size_t chol_smem = chol_bytes(rank), trsm_smem = trsm_bytes(rank);
  for (int pass = 0; pass < 2; ++pass) {
    dion_gram_kernel<<<dim3(unsigned(T * (T + 1) / 2), unsigned(plan.max_gchunks), nb), 256, 0,
                       stream>>>(c, pass);
    if (!launched()) return MAO_ERR_CUDA;
    dion_chol_kernel<<<nb, kCholThreads, chol_smem, stream>>>(c);
    if (!launched()) return MAO_ERR_CUDA;
    dion_trsm_kernel<<<dim3(unsigned(plan.max_rowtiles), nb), kTrsmThreads, trsm_smem, stream>>>(
        c, pass);
    if (!launched()) return MAO_ERR_CUDA;
  }
  // 4. R = B^T P (fp32)
  st = dion_tc(plan, ws, c.tR, 1, 1.0f, stream);
  if (st != MAO_OK) return st;
  // 5. Q = ColumnNormalize(R) (caller's Q), bf16 copies of Q and R
  dion_colnorm_kernel<<<dim3(unsigned(T), unsigned(plan.max_nchunks), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  dion_norm_kernel<<<nb, 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  dion_q_kernel<<<dim3(blocks(plan.max_qunits), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  // 6. M <- B - (1 - mu) P R^T ; X <- X - lr P Q^T (in place)
  st = dion_tc(plan, ws, c.tM, 2, -(1.0f - mu), stream);
  if (st != MAO_OK) return st;
  return dion_tc(plan, ws, c.tX, 3, -lr, stream);
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
  for (int b = 0; b < batch; ++b) {
    if (X[b].rows < 1 || X[b].cols < 1 || X[b].rows > (int64_t(1) << 31) ||
        X[b].cols > (int64_t(1) << 31))
      return 0;
    if (rank > std::min(X[b].rows, X[b].cols)) return 0;
  }
  return dion_workspace_size(X, batch, rank);
}

mao_status dion_step(const mao_mat* X, const mao_mat* M, const mao_mat* G, const mao_mat* Q,
                     float* const* P_out, int32_t batch, int32_t rank, float mu, float lr,
                     int32_t compute, void* workspace, size_t workspace_bytes, void* stream) {
  if (!X || !M || !G || !Q || batch < 1 || rank < 1 || rank > kMaxRank) return MAO_ERR_INVALID_ARG;
  if (!std::isfinite(mu) || !std::isfinite(lr)) return MAO_ERR_INVALID_ARG;
  if (compute != MAO_BF16) return MAO_ERR_UNSUPPORTED;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_mat(X[b]);
    if (st == MAO_OK) st = check_mat(M[b]);
    if (st == MAO_OK) st = check_mat(G[b]);
    if (st == MAO_OK) st = check_mat(Q[b]);
    if (st != MAO_OK) return st;
    const int64_t m = X[b].rows, n = X[b].cols;
    if (M[b].rows != m || M[b].cols != n || G[b].rows != m || G[b].cols != n)
      return MAO_ERR_INVALID_ARG;
    if (Q[b].dtype != MAO_F32 || Q[b].rows != n || Q[b].cols != rank) return MAO_ERR_INVALID_ARG;
    if (rank > std::min(m, n)) return MAO_ERR_INVALID_ARG;
    if (P_out && P_out[b] && reinterpret_cast<uintptr_t>(P_out[b]) % 4 != 0)
      return MAO_ERR_MISALIGNED;
  }
  if (batch > 65535) return MAO_ERR_UNSUPPORTED;
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < dion_workspace_size(X, batch, rank)) return MAO_ERR_WORKSPACE;
  return dion_run(X, M, G, Q, P_out, batch, rank, mu, lr, workspace,
                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
