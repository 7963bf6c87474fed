// One Dion step on the GPU ("대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습",
// algorithm section): for each parameter matrix X (m x n) with momentum M, gradient G and
// the previous right factor Q (n x r),
//
//   B = M + G                       stage kernel: bf16 copy Bw (and M <- B for an fp32 M)
//   P = orthonormalise(B Q)         tensor-core product (fp32 P), then Cholesky QR twice
//   R = B^T P                       tensor-core product (fp32 R)
//   Q <- ColumnNormalize(R)         column norms, then Q (fp32, caller) and bf16 copies
//   M <- B - (1 - mu) P R^T         tensor-core rank-r update (B read from M, or from Bw)
//   X <- X - lr P Q^T               tensor-core rank-r update, in place
//
// The orthonormal basis is the Q factor of the thin QR with a positive triangular
// diagonal, computed as Cholesky QR applied twice: S = P^T P, S = L L^T, P <- P W^T with
// W = L^-1 (the factorisation kernel also inverts L, so the product with P is one parallel
// multiply instead of a sequential substitution).
// The dense products (B Q, B^T P and the two rank-r updates) run on the same tcgen05 kernel
// as Newton–Schulz, over up to eight shape groups per launch. The Cholesky factorisation and
// its inverse run in fp32 on CUDA cores, one CTA per matrix. The two products of Cholesky QR
// run on the tensor cores from bf16 parts of their fp32 factors (x = hi + mid + lo with
// hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid)), fp32 accumulation:
//   Gram    S = P^T P from D = [P_hi P_mid]^T [P_hi P_mid P_lo]: hh + hm + mh + hl + lh + mm,
//           leaving out terms below 2^-26 of |P|^2, so the Cholesky factor is as good as
//           with an fp32 Gram (Cholesky QR needs kappa(P)^2 times the Gram's error < 1);
//   multiply P W^T (W = L^-1) = [P_hi P_hi P_mid] [W_hi W_lo W_hi]^T, about 2^-17 relative
//           (P enters the later products as bf16, 2^-9). Per-matrix
// descriptors live in a device table in the workspace (written by a set-up kernel), so a
// call of any size and any mix of shapes takes a fixed number of launches.
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
constexpr int kSetup = 96;        // table entries written per set-up launch (kernel parameters <= 32 KB)
constexpr int kCholThreads = 512;

// Everything the CUDA-core kernels need about one matrix slot.
struct DionSlot {
  void* M;
  const void* G;
  void* X;
  void* Xo;                         // the updated X (X itself, or the caller's X_out)
  float* Q;
  float* Pout;                      // optional copy of the final P (m x r, row stride r)
  __nv_bfloat16 *Bw, *Qw, *Rw, *Pw; // bf16 operands, rows of ldn / ldr elements
  float* Rf;                        // fp32 R [n][ldr]
  float* Sf;                        // S = P^T P in lower 32 x 32 blocks (layout of blk())
  __nv_bfloat16 *Ys, *Ys2;          // P in bf16 parts [m][4 ldr]: hi | hi | mid | lo (B Q_prev,
                                    // then after the first Cholesky QR pass)
  float* D;                         // Gram work product [2 ldr][3 ldr] (fp32)
  __nv_bfloat16* Wsp;               // L^-1 split [ldr][3 ldr]: hi | lo | hi (rows j, columns k)
  float* cn;                        // column norms of R: partial sums of squares [nrb][ldr]
                                    // (32 rows each, from the B^T P product), then r norms
  int64_t ldm, ldg, ldx, ldq, ldxo;
  int32_t m, n, ldn;
  int32_t dtm, dtg, dtx;
  int32_t flags_m, flags_x;
  int32_t nrb;                      // 32-row blocks of R (ceil(n / 32))
  int32_t vec;                      // M and G: bf16/f32 rows that allow 16-byte accesses
  int32_t qvec;                     // Q: 16-byte aligned rows (ldq a multiple of 4)
};

struct DionCommon {
  const DionSlot* slots;            // device table [count]
  OutEntry *tP, *tM, *tX;  // output tables of the tensor-core launches [count]
  int32_t r, ldr, count;
};


struct SetupParams {
  DionSlot s[kSetup];
  int32_t n, z0;
  DionCommon c;
};
static_assert(sizeof(SetupParams) <= 32000, "set-up parameters exceed the kernel parameter limit");

// ---------------------------------------------------------------- set-up

// CTA k writes slot z0 + k of the device table (one 4-byte word per thread: the parameter
// reads of a warp then differ only in the word, not the slot) and its three output entries:
// the final P when the caller asked for a copy of it, and the two in-place updates.
__global__ void __launch_bounds__(64) dion_setup_kernel(const __grid_constant__ SetupParams p) {
  const int k = blockIdx.x;
  const DionSlot& e = p.s[k];
  const int z = p.z0 + k;
  static_assert(sizeof(DionSlot) % 4 == 0 && sizeof(DionSlot) / 4 <= 128, "slot copy by words");
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&e);
  uint32_t* dst = reinterpret_cast<uint32_t*>(const_cast<DionSlot*>(p.c.slots) + z);
  for (int w = threadIdx.x; w < int(sizeof(DionSlot) / 4); w += 64) dst[w] = src[w];
  if (threadIdx.x != 0) return;
  OutEntry o = {};
  // the final P: the bf16 operand Pw, and the caller's fp32 copy if asked for
  o.out = e.Pw;
  o.ld = p.c.ldr;
  o.dtype = MAO_BF16;
  o.flags = OUT_VEC;
  if (e.Pout) {
    o.copy = e.Pout;
    o.copy_ld = p.c.r;
    o.copy_cols = p.c.r;
    if (reinterpret_cast<uintptr_t>(e.Pout) % 16 == 0 && p.c.r % 4 == 0) o.flags |= OUT_COPY_VEC;
  }
  p.c.tP[z] = o;
  o = OutEntry{};
  o.out = e.M;
  o.ld = e.ldm;
  o.dtype = e.dtm;
  o.flags = e.flags_m;
  if (e.dtm == MAO_BF16) {  // B was not written back to M: the update reads it from Bw
    o.src = e.Bw;
    o.src_ld = e.ldn;
  }
  p.c.tM[z] = o;
  // X <- X - lr P Q^T, written to Xo (reading X when Xo is another matrix)
  o.src = e.Xo != e.X ? e.X : nullptr;
  o.src_ld = e.Xo != e.X ? e.ldx : 0;
  o.out = e.Xo;
  o.ld = e.ldxo;
  o.dtype = e.dtx;
  o.flags = e.flags_x;
  p.c.tX[z] = o;
}

// Lets the next launch in the stream (a tensor-core product, launched with programmatic
// stream serialization) start its set-up on the SMs this grid leaves free; the product
// still waits for this grid's completion (griddepcontrol.wait) before it reads any result.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- B = M + G, Qw

__device__ __forceinline__ float round_to(float v, int32_t dt) {
  return dt == MAO_BF16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// Columns j0 .. j0 + 7 of row i of the caller's Q (zeros at and past r), 16 bytes at a time
// where the row allows it.
__device__ __forceinline__ void load_q8(const DionSlot& e, int r, int64_t i, int j0, float (&v)[8]) {
  const float* q = e.Q + i * e.ldq;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = j0 + 4 * h;
    if (e.qvec && j + 4 <= r) {
      const float4 x = *reinterpret_cast<const float4*>(q + j);
      v[4 * h] = x.x;
      v[4 * h + 1] = x.y;
      v[4 * h + 2] = x.z;
      v[4 * h + 3] = x.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[4 * h + k] = j + k < r ? q[j + k] : 0.0f;
    }
  }
}

__device__ __forceinline__ void store_q8(const DionSlot& e, int r, int64_t i, int j0, const float (&v)[8]) {
  float* q = e.Q + i * e.ldq;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = j0 + 4 * h;
    if (e.qvec && j + 4 <= r) {
      *reinterpret_cast<float4*>(q + j) = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (j + k < r) q[j + k] = v[4 * h + k];
    }
  }
}

// Qw = bf16(Q_prev), zero-padded to ldr columns: block qb of the slot's Q units (8 columns
// each), kStageUnits per thread.
__device__ __forceinline__ void stage_q_block(const DionCommon& c, const DionSlot& e, uint32_t qb);

// One unit of the general path: Bw(row, col0 .. col0 + 7), and M when it is fp32.
__device__ __forceinline__ void dion_stage_unit(const DionSlot& e, int64_t row, int64_t col0) {
  float b[8];
  if (e.vec && col0 + 8 <= e.n) {
    float mv[8], gv[8];
    load8(e.M, row * e.ldm + col0, e.dtm, mv);
    load8(e.G, row * e.ldg + col0, e.dtg, gv);
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = mv[k] + gv[k];
    if (e.dtm != MAO_BF16) store8(e.M, row * e.ldm + col0, e.dtm, b);
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = round_to(b[k], e.dtm);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t j = col0 + k;
      b[k] = 0.0f;
      if (j < e.n) {
        const float v = load_elem(e.M, row * e.ldm + j, e.dtm) + load_elem(e.G, row * e.ldg + j, e.dtg);
        if (e.dtm != MAO_BF16) store_elem(e.M, row * e.ldm + j, e.dtm, v);
        b[k] = round_to(v, e.dtm);
      }
    }
  }
  store8(e.Bw, row * e.ldn + col0, MAO_BF16, b);
}

// Units of 8 columns over the zero-padded rows of Bw; blockIdx.y = slot. Bw = bf16 of
// B = M + G rounded to M's dtype, and M <- B when M is fp32. A bf16 M is left as it is:
// Bw then holds B exactly, and the M update reads B from there (its output entry's source).
// kStageUnits units per thread, 256 kStageUnits per block (a thread's units are 256 apart,
// so each load instruction of a warp reads 512 contiguous bytes).
constexpr int kStageUnits = 4;

__global__ void __launch_bounds__(256) dion_stage_kernel(const __grid_constant__ DionCommon c) {
  allow_dependent_launch();
  const DionSlot& e = c.slots[blockIdx.y];
  const uint32_t upr = uint32_t(e.ldn) / 8;
  const uint32_t units = uint32_t(e.m) * upr;
  // blocks past the slot's B units convert Q_prev
  const uint32_t bblocks = (units + 256u * kStageUnits - 1) / (256u * kStageUnits);
  if (blockIdx.x >= bblocks) {
    stage_q_block(c, e, blockIdx.x - bblocks);
    return;
  }
  const uint32_t ub = blockIdx.x * (256u * kStageUnits) + threadIdx.x;
  if (ub >= units) return;
  if (e.vec && e.dtm == MAO_BF16 && e.dtg == MAO_BF16) {
    // bf16 M and G: every unit's loads are issued before any arithmetic; B = bf16(M + G)
    // as in dion_stage_unit
    uint4 mv[kStageUnits], gv[kStageUnits];
    uint32_t row[kStageUnits], col0[kStageUnits];
    bool live[kStageUnits], full[kStageUnits];
#pragma unroll
    for (int t = 0; t < kStageUnits; ++t) {
      const uint32_t u = ub + 256u * t;
      live[t] = u < units;
      row[t] = (live[t] ? u : 0u) / upr;
      col0[t] = ((live[t] ? u : 0u) - row[t] * upr) * 8u;
      full[t] = live[t] && int64_t(col0[t]) + 8 <= e.n;
      if (full[t]) {
        mv[t] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(e.M) +
                                                int64_t(row[t]) * e.ldm + col0[t]);
        gv[t] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(e.G) +
                                                     int64_t(row[t]) * e.ldg + col0[t]));
      }
    }
#pragma unroll
    for (int t = 0; t < kStageUnits; ++t) {
      if (!live[t]) continue;
      if (!full[t]) {
        dion_stage_unit(e, row[t], col0[t]);
        continue;
      }
      uint32_t* hm = reinterpret_cast<uint32_t*>(&mv[t]);
      const uint32_t* hg = reinterpret_cast<const uint32_t*>(&gv[t]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b =
            __floats2bfloat162_rn(__uint_as_float(hm[k] << 16) + __uint_as_float(hg[k] << 16),
                                  __uint_as_float(hm[k] & 0xFFFF0000u) + __uint_as_float(hg[k] & 0xFFFF0000u));
        hm[k] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(e.Bw + int64_t(row[t]) * e.ldn + col0[t]) = mv[t];
    }
    return;
  }
#pragma unroll 1
  for (int t = 0; t < kStageUnits; ++t) {
    const uint32_t u = ub + 256u * t;
    if (u >= units) break;
    const uint32_t row = u / upr;
    dion_stage_unit(e, row, int64_t(u - row * upr) * 8);
  }
}

__device__ __forceinline__ void stage_q_block(const DionCommon& c, const DionSlot& e, uint32_t qb) {
  const uint32_t upr = uint32_t(c.ldr) / 8;
  const uint32_t units = uint32_t(e.n) * upr;
#pragma unroll
  for (int t = 0; t < kStageUnits; ++t) {
    const uint32_t u = qb * (256u * kStageUnits) + 256u * t + threadIdx.x;
    if (u >= units) break;
    const uint32_t i = u / upr, j0 = (u - i * upr) * 8;
    float v[8];
    load_q8(e, c.r, i, int(j0), v);
    store8(e.Qw, size_t(i) * c.ldr + j0, MAO_BF16, v);
  }
}

// ------------------------------------------------------- Cholesky QR: S = P^T P

// Lower blocks of a matrix cut into 32 x 32 blocks, block (I, J) with I >= J at index
// I (I + 1) / 2 + J, each block 32 rows of kLd = 36 floats: rows start on 16-byte
// boundaries (broadcast row reads take 16 bytes at a time), a warp's column reads are
// contiguous, and 16-byte row reads of a quarter warp (lane = row) fall on distinct banks.
constexpr int kLd = 36;
constexpr int kBlk = 32 * kLd;  // floats of one block

__device__ __forceinline__ float* blk(float* A, int I, int J) {
  return A + (I * (I + 1) / 2 + J) * kBlk;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); bytes past `src_bytes`
// (0..16) are zero-filled and not read.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const uint32_t d = uint32_t(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Two floats rounded to bf16 (round to nearest even), the first in the low half.
__device__ __forceinline__ uint32_t bf16_pair(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}


// Factors the 32 x 32 diagonal block Ad = L L^T and forms D = L^-1 alongside, in registers:
// lane i holds row i of A (which becomes row i of L) and column i of D. Right-looking: at
// pivot j the pivot p = A_jj comes from lane j by a shuffle, every lane forms its
// L_ij = A_ij / sqrt(p) (lane j: sqrt(p) = p rsqrt(p)) and puts it into `col` (two
// alternating buffers in shared memory, lane i at position i - j + 31, so that the entries
// below the pivot start on a 16-byte boundary), then reads them back with 16-byte broadcast
// reads to update its row, A_ik -= L_ij L_kj for k > j, and its column c of D by forward
// substitution, D_jc = rhs_jc / L_jj and rhs_kc -= L_kj D_jc for k > j. One shuffle and one
// column broadcast per pivot serve both the factor and its inverse. The registers hold only
// the entries at and past the current pivot, moved down one place by each pivot's update,
// so the pivot loop is the same code for every j and stays rolled (its instructions come
// from the instruction cache after the first pivot, not from memory). Row j of D is written
// to Ad at pivot j (zeros above the diagonal). A pivot that is not positive is replaced by
// 1e-30 and reported.
__device__ __noinline__ bool chol_inv32(float* Ad, float* col, int lane) {
  float a[32], x[32];  // a[k]: A_lane,j+k; x[k]: rhs_j+k,lane (at pivot j)
#pragma unroll
  for (int q = 0; q < 32; q += 4) {
    const float4 v = ld4(Ad + lane * kLd + q);
    a[q] = q <= lane ? v.x : 0.0f;
    a[q + 1] = q + 1 <= lane ? v.y : 0.0f;
    a[q + 2] = q + 2 <= lane ? v.z : 0.0f;
    a[q + 3] = q + 3 <= lane ? v.w : 0.0f;
  }
#pragma unroll
  for (int k = 0; k < 32; ++k) x[k] = k == lane ? 1.0f : 0.0f;
  __syncwarp();  // every row is in registers before row 0 of D overwrites it
  bool bad = false;
#pragma unroll 1
  for (int j = 0; j < 32; ++j) {
    float p = __shfl_sync(0xFFFFFFFFu, a[0], j);
    if (!(p > 0.0f)) {
      bad = true;
      p = 1e-30f;
    }
    const float inv = rsqrtf(p);
    const float d = x[0] * inv;  // D_j,lane
    Ad[j * kLd + lane] = d;
    const float l = lane > j ? a[0] * inv : (lane == j ? p * inv : 0.0f);
    float* cb = col + 64 * (j & 1);
    cb[lane - j + 31] = l;  // L_ij at cb[32 + (i - j - 1)]
    __syncwarp();
    float c[32];
#pragma unroll
    for (int q = 0; q < 32; q += 4) {
      const float4 v = ld4(cb + 32 + q);
      c[q] = v.x;
      c[q + 1] = v.y;
      c[q + 2] = v.z;
      c[q + 3] = v.w;
    }
#pragma unroll
    for (int k = 0; k < 31; ++k) a[k] = __fmaf_rn(-l, c[k], a[k + 1]);
    a[31] = 0.0f;
#pragma unroll
    for (int k = 0; k < 31; ++k) x[k] = __fmaf_rn(-c[k], d, x[k + 1]);
    x[31] = 0.0f;
  }
  __syncwarp();
  return bad;
}

// L_IJ = A_IJ D_J^T (D_J = L_JJ^-1) for the rows [row0, row1) of block column J: warp w of
// nw takes rows row0 + w, row0 + w + nw, ...; lane = column, the lane's row of D_J held in
// registers across the rows.
__device__ __forceinline__ void chol_panel(float* A, int J, int row0, int row1, int w, int nw, int lane) {
  if (row0 + w >= row1) return;
  const float* Dj = blk(A, J, J) + lane * kLd;
  float4 d[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = ld4(Dj + 4 * q);
  for (int row = row0 + w; row < row1; row += nw) {
    float* Ap = blk(A, row >> 5, J) + (row & 31) * kLd;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = ld4(Ap + 4 * q);
      s0 = __fmaf_rn(v.x, d[q].x, s0);
      s1 = __fmaf_rn(v.y, d[q].y, s1);
      s0 = __fmaf_rn(v.z, d[q].z, s0);
      s1 = __fmaf_rn(v.w, d[q].w, s1);
    }
    __syncwarp();
    Ap[lane] = s0 + s1;
  }
}

// Rows r0 .. r0 + NR - 1 of A_IK -= L_IJ L_KJ^T (lane = column, the lane's row of L_KJ in
// registers, rows of L_IJ by 16-byte broadcast reads).
template <int NR>
__device__ __forceinline__ void chol_update(float* A, int J, int I, int K, int r0, int lane) {
  float4 lk[8];
  const float* Lk = blk(A, K, J) + lane * kLd;
#pragma unroll
  for (int q = 0; q < 8; ++q) lk[q] = ld4(Lk + 4 * q);
  const float* Li = blk(A, I, J) + r0 * kLd;
  float* Ab = blk(A, I, K) + r0 * kLd;
#pragma unroll
  for (int tt = 0; tt < NR; ++tt) {
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 l = ld4(Li + tt * kLd + 4 * q);
      s0 = __fmaf_rn(l.x, lk[q].x, s0);
      s1 = __fmaf_rn(l.y, lk[q].y, s1);
      s0 = __fmaf_rn(l.z, lk[q].z, s0);
      s1 = __fmaf_rn(l.w, lk[q].w, s1);
    }
    Ab[tt * kLd + lane] -= s0 + s1;
  }
}

// Block row K of W = L^-1 to global memory as the bf16 operand of the multiply P W^T on
// the tensor cores: row j holds hi(W_j) | lo(W_j) | hi(W_j), ldr columns each,
// lo = bf16(w - hi). Block (K, J) comes from Wr + J kBlk for J < K and is D_K = Dk for J = K;
// zeros above the diagonal. With `last`, the rows past the 32 nb rows of the blocks follow as
// the identity. Thread t of nt. Not inlined (one copy of the code for all block rows).
__device__ __noinline__ void chol_write_w(const float* Wr, const float* Dk, __nv_bfloat16* Wsp, int K, int nb,
                                             int ldr, bool last, int t, int nt) {
  const int q8 = ldr / 8, nbw32 = 32 * nb;
  const int j0 = 32 * K, j1 = last ? ldr : 32 * (K + 1);
  for (int q = t; q < (j1 - j0) * q8; q += nt) {
    const int dj = q / q8, j = j0 + dj, k0 = (q - dj * q8) * 8;
    float w[8], lo[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u;
      float val;
      if (j < nbw32 && k < nbw32) {
        const int J = k >> 5;
        const float* src = J < K ? Wr + J * kBlk : Dk;
        val = J <= K && k <= j ? src[(j & 31) * kLd + (k & 31)] : 0.0f;
      } else {
        val = j == k ? 1.0f : 0.0f;
      }
      w[u] = val;
      lo[u] = val - __bfloat162float(__float2bfloat16_rn(val));
    }
    const uint4 h = make_uint4(bf16_pair(w[0], w[1]), bf16_pair(w[2], w[3]), bf16_pair(w[4], w[5]),
                               bf16_pair(w[6], w[7]));
    const uint4 l = make_uint4(bf16_pair(lo[0], lo[1]), bf16_pair(lo[2], lo[3]), bf16_pair(lo[4], lo[5]),
                               bf16_pair(lo[6], lo[7]));
    __nv_bfloat16* row = Wsp + size_t(j) * 3 * ldr;
    *reinterpret_cast<uint4*>(row + k0) = h;
    *reinterpret_cast<uint4*>(row + ldr + k0) = l;
    *reinterpret_cast<uint4*>(row + 2 * ldr + k0) = h;
  }
}

// Register-tiled products of 32 x 32 blocks (row stride kLd) for one warp. Lane (ri, ck) =
// (lane & 7, lane >> 3) holds rows r0 + ri + 8u (u < NU) of the result. Every read of the
// operands happens before any write of C, so C may be X (each warp writes only its own rows).

// C = alpha X Y^T (+ C with ACC), the product over the columns of X and Y (both row-major):
// columns ck + 4v (v < 8) of the lane's rows. The X and Y row reads (16 bytes) and the
// entries' reads and writes are free of bank conflicts.
template <int NU, bool ACC>
__device__ __forceinline__ void blk_nt(const float* X, const float* Y, float* C, int r0, float alpha,
                                       int lane) {
  const int ri = lane & 7, ck = lane >> 3;
  float acc[NU][8];
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[u][v] = 0.0f;
#pragma unroll 2
  for (int j = 0; j < 32; j += 4) {
    float4 x[NU], y[8];
#pragma unroll
    for (int u = 0; u < NU; ++u) x[u] = ld4(X + (r0 + ri + 8 * u) * kLd + j);
#pragma unroll
    for (int v = 0; v < 8; ++v) y[v] = ld4(Y + (ck + 4 * v) * kLd + j);
#pragma unroll
    for (int u = 0; u < NU; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        float a = acc[u][v];
        a = __fmaf_rn(x[u].x, y[v].x, a);
        a = __fmaf_rn(x[u].y, y[v].y, a);
        a = __fmaf_rn(x[u].z, y[v].z, a);
        a = __fmaf_rn(x[u].w, y[v].w, a);
        acc[u][v] = a;
      }
  }
  __syncwarp();
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      float* c = C + (r0 + ri + 8 * u) * kLd + ck + 4 * v;
      *c = ACC ? __fmaf_rn(alpha, acc[u][v], *c) : alpha * acc[u][v];
    }
  __syncwarp();
}

// C = alpha X Y (+ C with ACC), the product over X's columns and Y's rows: columns
// 8 ck .. 8 ck + 7 of the lane's rows (16-byte reads and writes).
template <int NU, bool ACC>
__device__ __forceinline__ void blk_nn(const float* X, const float* Y, float* C, int r0, float alpha,
                                       int lane) {
  const int ri = lane & 7, ck = lane >> 3;
  float acc[NU][8];
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[u][v] = 0.0f;
#pragma unroll 2
  for (int k = 0; k < 32; k += 4) {
    float4 x[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) x[u] = ld4(X + (r0 + ri + 8 * u) * kLd + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 y0 = ld4(Y + (k + kk) * kLd + 8 * ck), y1 = ld4(Y + (k + kk) * kLd + 8 * ck + 4);
      const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const float xv = kk == 0 ? x[u].x : kk == 1 ? x[u].y : kk == 2 ? x[u].z : x[u].w;
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = __fmaf_rn(xv, yv[v], acc[u][v]);
      }
    }
  }
  __syncwarp();
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    float* c = C + (r0 + ri + 8 * u) * kLd + 8 * ck;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 o = make_float4(alpha * acc[u][4 * h], alpha * acc[u][4 * h + 1], alpha * acc[u][4 * h + 2],
                             alpha * acc[u][4 * h + 3]);
      if (ACC) {
        const float4 old = ld4(c + 4 * h);
        o = make_float4(old.x + o.x, old.y + o.y, old.z + o.z, old.w + o.w);
      }
      *reinterpret_cast<float4*>(c + 4 * h) = o;
    }
  }
  __syncwarp();
}

// Inverse step K, part 1, 2 or 3 (see the kernel below), one block per item; nb - 1 - K
// block rows lie below K. Not inlined: the loop over the block columns
// and the last two steps share its code, which is then fetched from memory once.
__device__ __noinline__ void chol_inv_item(float* A, float* Wr, int part, int K, int item, int lane) {
  const int b = item;
  if (part == 1) {  // item < K: W_KJ = -D_K T_KJ into Wr
    blk_nn<4, false>(blk(A, K, K), blk(A, K, b), Wr + b * kBlk, 0, -1.0f, lane);
  } else if (part == 2) {  // item < (nb - 1 - K) K: T_IJ += L_IK W_KJ
    const int I = K + 1 + b / K, J = b % K;
    blk_nn<4, true>(blk(A, I, K), Wr + J * kBlk, blk(A, I, J), 0, 1.0f, lane);
  } else {  // item < nb - 1 - K: T_IK = L_IK D_K (in place)
    const int I = K + 1 + b;
    blk_nn<4, false>(blk(A, I, K), blk(A, K, K), blk(A, I, K), 0, 1.0f, lane);
  }
}

// Trailing work of block column J, one block per item: the panel L_IJ = A_IJ D_J^T
// (I = J + 2 + item, item < t), or (trailing) A_IK -= L_IJ L_KJ^T over the t blocks of
// column J + 1 below the diagonal and then the triangle K >= J + 2
// (item < t + t (t + 1) / 2). Not inlined (one copy of the code).
__device__ __noinline__ void chol_trail_item(float* A, bool panel, int J, int t, int item, int lane) {
  int b = item;
  if (panel) {
    const int I = J + 2 + b;
    blk_nt<4, false>(blk(A, I, J), blk(A, J, J), blk(A, I, J), 0, 1.0f, lane);
    return;
  }
  int I, K;
  if (b < t) {
    I = J + 2 + b;
    K = J + 1;
  } else {
    b -= t;
    I = 0;
    K = b;
    while (K > I) {
      K -= I + 1;
      ++I;
    }
    I += J + 2;
    K += J + 2;
  }
  blk_nt<4, true>(blk(A, I, J), blk(A, K, J), blk(A, I, K), 0, -1.0f, lane);
}

// One CTA per slot: S = L L^T (blocked right-looking Cholesky, 32 x 32 blocks in shared
// memory) and W = L^-1, written to e.Wsp as the split bf16 operand of the multiply P W^T.
// After block J's factorisation the diagonal block holds D_J = L_JJ^-1, which is all that
// later steps need of it. W is formed right-looking as well: block (I, J) of the lower
// triangle passes from A_IJ to L_IJ (panel) and then to the sum
// T_IJ = sum_{K = J .. } L_IK W_KJ over the block rows K of W final so far (starting with
// L_IJ D_J); W_IJ = -D_I T_IJ once all K < I have been added. Inverse step K, once block row
// K of the sums and block column K of L are final:
//   (1) W_KJ = -D_K T_KJ for J < K, into the row buffer Wr (block row K of W is then final
//       and goes to global memory from there),
//   (2) T_IJ += L_IK W_KJ for I > K, J < K,
//   (3) T_IK = L_IK D_K for I > K (in place of L_IK, after (2) has read it).
// For each block column J of the factorisation:
//   critical path (all warps): block row J + 1 of the panel, L_J+1,J = A_J+1,J D_J^T, then
//   the diagonal block A_J+1,J+1 -= L_J+1,J L_J+1,J^T; then warp 0 factors and inverts the
//   diagonal block J + 1 (chol_inv32) while the other warps finish the panel (L_IJ for
//   I >= J + 2), update the trailing blocks A_IK, J + 1 <= K <= I, I >= J + 2, and take
//   inverse step J - 1 (one block per item, register-tiled).
// The last two inverse steps run on all warps at the end. S arrives in this block layout
// (the assemble kernel writes it so). Rows and columns past r are the identity. A pivot
// that is not positive sets the device error word (P had dependent columns).
__global__ void __launch_bounds__(kCholThreads, 1) dion_chol_kernel(const __grid_constant__ DionCommon c) {
  extern __shared__ __align__(16) float sm[];
  __shared__ __align__(16) float col[128];  // chol_inv32's column broadcast (two buffers)
  allow_dependent_launch();
  const DionSlot& e = c.slots[blockIdx.x];
  const int r = c.r, ldr = c.ldr;
  const int nb = (r + 31) / 32;
  const int nlow = nb * (nb + 1) / 2;
  float* A = sm;                 // nlow blocks
  float* Wr = A + nlow * kBlk;   // nb - 1 blocks: the block row of W of the current inverse step
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int kWarps = kCholThreads / 32;
  constexpr int kHelpers = kWarps - 1;  // every warp but warp 0
  // the lower blocks of S (their Gram entries past r are zero), then ones on the diagonal
  // past r
  for (int q = threadIdx.x; q < nlow * kBlk / 4; q += kCholThreads)
    cp_async16(A + 4 * q, e.Sf + 4 * q, 16);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  for (int i = r + int(threadIdx.x); i < 32 * nb; i += kCholThreads)
    blk(A, i / 32, i / 32)[(i % 32) * kLd + (i % 32)] = 1.0f;
  auto inv1 = [&](int K, int item) { chol_inv_item(A, Wr, 1, K, item, lane); };
  auto inv2 = [&](int K, int item) { chol_inv_item(A, Wr, 2, K, item, lane); };
  auto inv3 = [&](int K, int item) { chol_inv_item(A, Wr, 3, K, item, lane); };
  __syncthreads();
  if (warp == 0 && chol_inv32(blk(A, 0, 0), col, lane) && lane == 0) atomicOr(&g_dion_error, 1u);
  __syncthreads();
  for (int J = 0; J + 1 < nb; ++J) {
    // the critical path: block row J + 1 of the panel (two rows per warp), then the
    // diagonal block J + 1 (two rows per warp)
    chol_panel(A, J, 32 * (J + 1), 32 * (J + 2), warp, kWarps, lane);
    __syncthreads();
    chol_update<2>(A, J, J + 1, J + 1, 2 * warp, lane);
    __syncthreads();
    if (warp == 0) {
      if (chol_inv32(blk(A, J + 1, J + 1), col, lane) && lane == 0) atomicOr(&g_dion_error, 1u);
    } else {
      // the other warps, numbered h = 0 .. kHelpers - 1 (sharing warp 0's sub-partition
      // slows the factorisation less than leaving three warps idle)
      const int h = warp - 1;
      auto hsync = [] { asm volatile("bar.sync 1, %0;" ::"r"(32 * kHelpers) : "memory"); };
      const int K = J - 1;       // inverse step taken in this block column
      const int t = nb - J - 2;  // block rows below J + 1
      // the rest of block column J of the panel; inverse step K part (1)
      const int np = t, n1 = K > 0 ? K : 0;
      for (int item = h; item < np + n1; item += kHelpers) {
        if (item < np) chol_trail_item(A, true, J, t, item, lane);
        else inv1(K, item - np);
      }
      hsync();
      // trailing blocks: t blocks of column J + 1 below the diagonal, then the triangle
      // K' >= J + 2; inverse step K part (2); block row K of W to global memory
      const int nu = t + t * (t + 1) / 2, n2 = K > 0 ? (nb - 1 - K) * K : 0;
      for (int item = h; item < nu + n2; item += kHelpers) {
        if (item < nu) chol_trail_item(A, false, J, t, item, lane);
        else inv2(K, item - nu);
      }
      if (K >= 0) chol_write_w(Wr, blk(A, K, K), e.Wsp, K, nb, ldr, false, h * 32 + lane, 32 * kHelpers);
      hsync();
      if (K >= 0)
        for (int item = h; item < nb - 1 - K; item += kHelpers) inv3(K, item);
    }
    __syncthreads();
  }
  // inverse steps nb - 2 and nb - 1 on all warps
  const int K = nb - 2;
  if (K >= 0) {
    for (int item = warp; item < K; item += kWarps) inv1(K, item);
    __syncthreads();
    for (int item = warp; item < K; item += kWarps) inv2(K, item);
    chol_write_w(Wr, blk(A, K, K), e.Wsp, K, nb, ldr, false, threadIdx.x, kCholThreads);
    __syncthreads();
    if (warp < 1) inv3(K, warp);
    __syncthreads();
  }
  for (int item = warp; item < nb - 1; item += kWarps) inv1(nb - 1, item);
  __syncthreads();
  chol_write_w(Wr, blk(A, nb - 1, nb - 1), e.Wsp, nb - 1, nb, ldr, true, threadIdx.x, kCholThreads);
}

// S = P^T P from the Gram work product D = [hi | mid]^T [hi | mid | lo] (rows: hi, then mid
// from row ldr; columns: hi, mid from ldr, lo from 2 ldr):
//   S = hi^T hi + hi^T mid + mid^T hi + hi^T lo + lo^T hi + mid^T mid,
// summed smallest first in a fixed order, into the lower 32 x 32 blocks the Cholesky kernel
// reads (entries at or past r are zero). The terms left out (mid^T lo, lo^T mid, lo^T lo) are
// below 2^-26 of |P|^2. mid^T hi is read from its own rows of D (D[ldr + i][k]); lo^T hi,
// which D holds only as hi^T lo, is read transposed. One block per 32 x 32 block of S
// (blockIdx.x), four consecutive entries of one row per thread: five 16-byte loads and four
// scalar ones for four entries.
__global__ void __launch_bounds__(256) dion_assemble_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.y];
  const int r = c.r, ldr = c.ldr;
  const int64_t ldd = 3 * int64_t(ldr);
  int b = blockIdx.x, I = 0;
  while (b > I) { b -= I + 1; ++I; }
  const int J = b, ii = threadIdx.x >> 3, k4 = 4 * (threadIdx.x & 7);
  const int i = 32 * I + ii, k = 32 * J + k4;
  float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (i < r && k < r) {
    const float* D = e.D;
    const float* Dh = D + i * ldd + k;           // row i (hi): hh | hm | hl
    const float* Dm = D + (ldr + i) * ldd + k;   // row ldr + i (mid): mh | mm
    const float4 hh = ld4(Dh), hm = ld4(Dh + ldr), hl = ld4(Dh + 2 * ldr);
    const float4 mh = ld4(Dm), mm = ld4(Dm + ldr);
    float lh[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) lh[t] = k + t < r ? D[(k + t) * ldd + 2 * ldr + i] : 0.0f;
    const float a[4] = {hh.x, hh.y, hh.z, hh.w}, bm[4] = {hm.x, hm.y, hm.z, hm.w};
    const float cl[4] = {hl.x, hl.y, hl.z, hl.w}, dm[4] = {mh.x, mh.y, mh.z, mh.w};
    const float em[4] = {mm.x, mm.y, mm.z, mm.w};
    float o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      o[t] = k + t < r ? (((em[t] + cl[t]) + lh[t]) + (bm[t] + dm[t])) + a[t] : 0.0f;
    v = make_float4(o[0], o[1], o[2], o[3]);
  }
  *reinterpret_cast<float4*>(blk(e.Sf, I, J) + ii * kLd + k4) = v;
}

// ------------------------------------------------------ R -> Q = ColumnNormalize(R)

// Reciprocal column norms: the 32-row partial sums of squares (written by the B^T P
// product's epilogue) added up, then 1 / sqrt (0 for a zero column); they go after the
// partials (e.cn + nrb * ldr). Grid (ldr / 32, slots): 32 columns per block, the row
// blocks dealt to 8 warps (b = warp, warp + 8, ...) and the 8 warps' sums added in a fixed
// order.
__global__ void __launch_bounds__(256) dion_norm_kernel(const __grid_constant__ DionCommon c) {
  const DionSlot& e = c.slots[blockIdx.y];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int j = int(blockIdx.x) * 32 + lane;
  float ss = 0.0f;
#pragma unroll 4
  for (int b = w; b < e.nrb; b += 8) ss += e.cn[size_t(b) * c.ldr + j];
  __shared__ float part[8][32];
  part[w][lane] = ss;
  __syncthreads();
  if (w == 0 && j < c.r) {
    float t = part[0][lane];
#pragma unroll
    for (int q = 1; q < 8; ++q) t += part[q][lane];
    e.cn[size_t(e.nrb) * c.ldr + j] = t > 0.0f ? 1.0f / sqrtf(t) : 0.0f;
  }
}

// Q = R / ||R_:j|| (times the reciprocal norm; a zero column stays zero) into the caller's
// Q, and the bf16 copies Qw, Rw; 8 columns per thread, 16-byte accesses.
__global__ void __launch_bounds__(256) dion_q_kernel(const __grid_constant__ DionCommon c) {
  allow_dependent_launch();
  const DionSlot& e = c.slots[blockIdx.y];
  const uint32_t upr = uint32_t(c.ldr) / 8;
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= uint32_t(e.n) * upr) return;
  const uint32_t i = u / upr, j0 = (u - i * upr) * 8;
  const float* rn = e.cn + size_t(e.nrb) * c.ldr;
  const float4* rp = reinterpret_cast<const float4*>(e.Rf + size_t(i) * c.ldr + j0);
  const float4 r0 = rp[0], r1 = rp[1];
  const float raw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  float rv[8], qv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int j = int(j0) + k;
    rv[k] = j < c.r ? raw[k] : 0.0f;
    qv[k] = j < c.r ? rv[k] * rn[j] : 0.0f;
  }
  store_q8(e, c.r, i, int(j0), qv);
  store8(e.Qw, size_t(i) * c.ldr + j0, MAO_BF16, qv);
  store8(e.Rw, size_t(i) * c.ldr + j0, MAO_BF16, rv);
}

// ----------------------------------------------------------------- orchestration

struct DionGroup {
  int64_t m, n;
  int32_t count, slot0;
  size_t off_bw, off_qw, off_rw, off_pw, off_rf, off_sf, off_ys, off_ys2, off_d, off_wsp, off_cn;
};

struct DionPlan {
  std::vector<DionGroup> groups;
  std::vector<int> input_of;  // slot -> caller's index
  int64_t r = 0, ldr = 0;
  size_t off_slots = 0, off_tables = 0, total = 0;
  int64_t max_units = 0, max_qunits = 0;
  int64_t max_stage_blocks = 0;  // B units, then Q units, of the largest slot
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
  plan.off_tables = take(3 * sizeof(OutEntry) * size_t(batch));
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
    const size_t nrb = size_t(ceil_div(g.n, 32));
    g.off_bw = take(c * m * ldn * 2);
    g.off_qw = take(c * n * ldr * 2);
    g.off_rw = take(c * n * ldr * 2);
    g.off_pw = take(c * m * ldr * 2);
    g.off_rf = take(c * n * ldr * 4);
    const size_t nsb = (ldr / 32) * (ldr / 32 + 1) / 2;  // lower 32 x 32 blocks of S
    g.off_sf = take(c * nsb * kBlk * 4);
    g.off_ys = take(c * m * 4 * ldr * 2);
    g.off_ys2 = take(c * m * 4 * ldr * 2);
    g.off_d = take(c * 2 * ldr * 3 * ldr * 4);
    g.off_wsp = take(c * ldr * 3 * ldr * 2);
    g.off_cn = take(c * (nrb * ldr + r) * 4);
    for (int b : mem) plan.input_of.push_back(b);
    slot += g.count;
    plan.max_units = std::max<int64_t>(plan.max_units, g.m * int64_t(ldn / 8));
    plan.max_stage_blocks = std::max<int64_t>(
        plan.max_stage_blocks, ceil_div(g.m * int64_t(ldn / 8), 256 * kStageUnits) +
                                   ceil_div(g.n * int64_t(ldr / 8), 256 * kStageUnits));
    plan.max_qunits = std::max<int64_t>(plan.max_qunits, g.n * int64_t(ldr / 8));
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
// op: 0 = P = B Q, 1 = R = B^T P, 2 = M update (P R^T), 3 = X update (P Q^T), 4 = the multiply
// P W^T and 5 = the Gram product of Cholesky QR pass `pass` (P's parts from Ys, then Ys2).
// B Q_prev, R, the Gram products and the multiplies go to workspace buffers through bulk
// stores (eight epilogue warps); only the final P with a caller's copy, and the updates, go
// through the slots' output entries (`table`).
// op 6: both in-place updates in one launch (M with alpha through table[slot], X with alpha2
// through table[batch + slot]), so that their tiles share the rounds.
mao_status dion_tc(const DionPlan& plan, uint8_t* ws, const OutEntry* table, int op, float alpha,
                   cudaStream_t stream, int pass = 0, float alpha2 = 0.0f) {
  const int64_t r = plan.r, ldr = plan.ldr;
  const int32_t batch = int32_t(plan.input_of.size());
  // The kernel deals tiles to CTA pairs in rounds, every other one reversed; listing the groups with
  // the deepest products (the most k-blocks per tile) first spreads the long tiles over the
  // pairs before the short ones fill the gaps.
  std::vector<std::pair<size_t, int>> order;  // (group, product) in launch order
  for (size_t i = 0; i < plan.groups.size(); ++i) order.push_back({i, op == 6 ? 2 : op});
  if (op == 6)
    for (size_t i = 0; i < plan.groups.size(); ++i) order.push_back({i, 3});
  auto depth = [&](const std::pair<size_t, int>& it) {
    const DionGroup& g = plan.groups[it.first];
    switch (it.second) {
      case 0: return g.n;
      case 1: return g.m;
      case 4: return 3 * ldr;
      case 5: return g.m;
      default: return r;
    }
  };
  std::stable_sort(order.begin(), order.end(),
                   [&](const std::pair<size_t, int>& x, const std::pair<size_t, int>& y) {
                     return depth(x) > depth(y);
                   });
  const bool update = op == 2 || op == 3 || op == 6;
  for (size_t g0 = 0; g0 < order.size(); g0 += tc::MAX_GROUPS) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.stage = update ? TC_UPDATE : NS_APPLY;
    p.a = alpha;
    p.scale = nullptr;
    p.out_table = table;
    p.timeout_ns = wait_limit_ns();
    p.snake = 1;  // tiles of mixed depths, deepest groups first
    int64_t tiles = 0;
    for (size_t gi = g0; gi < order.size() && p.ngroups < tc::MAX_GROUPS; ++gi) {
      const DionGroup& g = plan.groups[order[gi].first];
      const int gop = order[gi].second;  // this group's product
      TcGroup& G = p.g[p.ngroups++];
      const int64_t ldn = round_up(g.n, tc::LD_ALIGN);
      const void *A, *B;
      int64_t rowsA, ldA, rowsB, ldB, colsA = -1, colsB = -1;
      switch (gop) {
        case 0:  // (m x n)(n x ldr): Bw K-major, Qw MN-major (zeros past r)
          A = ws + g.off_bw; rowsA = g.m; ldA = ldn; G.a_mn = 0;
          B = ws + g.off_qw; rowsB = g.n; ldB = ldr; G.b_mn = 1;
          G.M = int32_t(g.m); G.N = int32_t(ldr); G.K = int32_t(g.n);
          break;
        case 1:  // (n x m)(m x ldr): Bw MN-major, Pw MN-major (zeros past r)
          A = ws + g.off_bw; rowsA = g.m; ldA = ldn; G.a_mn = 1;
          B = ws + g.off_pw; rowsB = g.m; ldB = ldr; G.b_mn = 1;
          G.M = int32_t(g.n); G.N = int32_t(ldr); G.K = int32_t(g.m);
          break;
        case 4:  // (m x 3 ldr)(3 ldr x ldr): [P_hi P_hi P_mid] [W_hi W_lo W_hi]^T, both K-major
          A = ws + (pass == 0 ? g.off_ys : g.off_ys2); rowsA = g.m; ldA = 4 * ldr; colsA = 3 * ldr;
          G.a_mn = 0;
          B = ws + g.off_wsp; rowsB = ldr; ldB = 3 * ldr; G.b_mn = 0;
          G.M = int32_t(g.m); G.N = int32_t(ldr); G.K = int32_t(3 * ldr);
          break;
        case 5:  // (2 ldr x m)(m x 3 ldr): [P_hi P_mid]^T [P_hi P_mid P_lo], both MN-major
          A = ws + (pass == 0 ? g.off_ys : g.off_ys2) + ldr * 2; rowsA = g.m; ldA = 4 * ldr;
          colsA = 2 * ldr; G.a_mn = 1;
          B = static_cast<const uint8_t*>(A); rowsB = g.m; ldB = 4 * ldr; colsB = 3 * ldr; G.b_mn = 1;
          G.M = int32_t(2 * ldr); G.N = int32_t(3 * ldr); G.K = int32_t(g.m);
          break;
        default:  // (m x r)(r x n): Pw K-major, Rw / Qw K-major
          A = ws + g.off_pw; rowsA = g.m; ldA = ldr; G.a_mn = 0;
          B = ws + (gop == 2 ? g.off_rw : g.off_qw); rowsB = g.n; ldB = ldr; G.b_mn = 0;
          G.M = int32_t(g.m); G.N = int32_t(g.n); G.K = int32_t(r);
          break;
      }
      G.count = g.count;
      // the X update's entries follow the M update's in the combined launch's table
      G.slot0 = g.slot0 + (op == 6 && gop == 3 ? batch : 0);
      G.alpha = op == 6 && gop == 3 ? alpha2 : alpha;
      G.orig_cols = G.N;
      // workspace outputs: B Q_prev and the first pass's P W^T as the bf16 parts of the next
      // Cholesky QR pass, the final P W^T as Pw (bf16) unless the caller wants a copy of P,
      // R and the Gram product in fp32
      const bool ws_out = op == 0 || op == 1 || op == 5 || (op == 4 && (pass == 0 || !table));
      G.final_out = ws_out ? 0 : 1;
      mao_status st = tc_encode_map(&G.tmA, A, rowsA, ldA, g.count, colsA);
      if (st == MAO_OK) st = tc_encode_map(&G.tmB, B, rowsB, ldB, g.count, colsB);
      if (st == MAO_OK && ws_out) {
        const int64_t rows = G.M, ld = op == 0 || op == 4 ? (pass == 0 ? 4 * ldr : ldr) : G.N;
        G.out = ws + (op == 0 ? g.off_ys : op == 1 ? g.off_rf : op == 5 ? g.off_d
                      : pass == 0 ? g.off_ys2 : g.off_pw);
        G.out_ld = ld;
        G.out_mstride = rows * ld;
        G.out_kind = op == 1 ? OUTK_F32_COLSQ : op == 5 ? OUTK_F32
                     : (op == 0 || pass == 0) ? OUTK_PARTS : OUTK_BF16;
        if (op == 1) {  // R's 32-row column sums of squares into the norm partials
          const int64_t nrb = ceil_div(g.n, 32);
          G.colsq = reinterpret_cast<float*>(ws + g.off_cn);
          G.colsq_mstride = nrb * ldr + r;
          G.colsq_ld = int32_t(ldr);
        }
        st = op == 1 || op == 5 ? tc_encode_store_map_f32(&G.tmOR, G.out, rows, ld, g.count)
                                : tc_encode_store_map(&G.tmOR, G.out, rows, ld, g.count);
      }
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
                    const mao_mat* X_out, float* const* P_out, int32_t batch, int32_t rank,
                    float mu, float lr, void* workspace, cudaStream_t stream) {
  DionPlan plan;
  make_dion_plan(X, batch, rank, plan);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  DionCommon c;
  c.slots = reinterpret_cast<const DionSlot*>(ws + plan.off_slots);
  OutEntry* tables = reinterpret_cast<OutEntry*>(ws + plan.off_tables);
  c.tP = tables;
  c.tM = tables + batch;
  c.tX = tables + 2 * batch;
  c.r = rank;
  c.ldr = int32_t(plan.ldr);
  c.count = batch;

  static std::once_flag attr_once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  cudaError_t attr_err = cudaSuccess;
  auto chol_bytes = [](int rk) {  // the lower blocks and one block row of W
    const size_t nbk = size_t(ceil_div(rk, 32));
    return sizeof(float) * size_t(kBlk) * (nbk * (nbk + 1) / 2 + nbk - 1);
  };
  const size_t chol_max = chol_bytes(kMaxRank);
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(dion_chol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(chol_max));
  });
  if (attr_err != cudaSuccess) return MAO_ERR_CUDA;
  auto launched = [stream] {
    profile_after_launch(stream);
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
      e.Xo = X_out ? X_out[b].data : X[b].data;
      e.Q = reinterpret_cast<float*>(Q[b].data);
      e.Pout = P_out ? P_out[b] : nullptr;
      e.Bw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_bw) + size_t(k) * g.m * ldn;
      e.Qw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_qw) + size_t(k) * g.n * plan.ldr;
      e.Rw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_rw) + size_t(k) * g.n * plan.ldr;
      e.Pw = reinterpret_cast<__nv_bfloat16*>(ws + g.off_pw) + size_t(k) * g.m * plan.ldr;
      e.Rf = reinterpret_cast<float*>(ws + g.off_rf) + size_t(k) * g.n * plan.ldr;
      e.nrb = int32_t(ceil_div(g.n, 32));
      const size_t nsb = size_t(plan.ldr / 32) * size_t(plan.ldr / 32 + 1) / 2;
      e.Sf = reinterpret_cast<float*>(ws + g.off_sf) + size_t(k) * nsb * kBlk;
      e.Ys = reinterpret_cast<__nv_bfloat16*>(ws + g.off_ys) + size_t(k) * g.m * 4 * plan.ldr;
      e.Ys2 = reinterpret_cast<__nv_bfloat16*>(ws + g.off_ys2) + size_t(k) * g.m * 4 * plan.ldr;
      e.D = reinterpret_cast<float*>(ws + g.off_d) + size_t(k) * 2 * plan.ldr * 3 * plan.ldr;
      e.Wsp = reinterpret_cast<__nv_bfloat16*>(ws + g.off_wsp) + size_t(k) * plan.ldr * 3 * plan.ldr;
      e.cn = reinterpret_cast<float*>(ws + g.off_cn) + size_t(k) * (e.nrb * plan.ldr + rank);
      e.ldm = M[b].ld;
      e.ldg = G[b].ld;
      e.ldx = X[b].ld;
      e.ldxo = X_out ? X_out[b].ld : X[b].ld;
      e.ldq = Q[b].ld;
      e.m = int32_t(g.m);
      e.n = int32_t(g.n);
      e.ldn = int32_t(ldn);
      e.dtm = M[b].dtype;
      e.dtg = G[b].dtype;
      e.dtx = X[b].dtype;
      e.flags_m = out_flags(M[b]);
      e.flags_x = out_flags(X[b]) & (X_out ? out_flags(X_out[b]) : ~0);
      e.vec = vec8_ok(M[b]) && vec8_ok(G[b]) ? 1 : 0;
      e.qvec = (reinterpret_cast<uintptr_t>(Q[b].data) % 16 == 0 && Q[b].ld % 4 == 0) ? 1 : 0;
    }
  }
  for (int z0 = 0; z0 < batch; z0 += kSetup) {
    SetupParams sp;
    memset(&sp, 0, sizeof(sp));
    sp.n = std::min(kSetup, batch - z0);
    sp.z0 = z0;
    sp.c = c;
    for (int k = 0; k < sp.n; ++k) sp.s[k] = slots[z0 + k];
    profile_before_launch(stream, MAO_PROF_DION_SETUP);
    dion_setup_kernel<<<unsigned(sp.n), 64, 0, stream>>>(sp);
    if (!launched()) return MAO_ERR_CUDA;
  }
  const unsigned nb = unsigned(batch);
  auto blocks = [](int64_t units) { return unsigned(ceil_div(units, 256)); };
  // 1. B = M + G (M <- B), Bw; Qw = bf16(Q_prev)
  profile_before_launch(stream, MAO_PROF_DION_STAGE);
  dion_stage_kernel<<<dim3(unsigned(plan.max_stage_blocks), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  // 2. P = B Q_prev, as the bf16 parts Ys
  mao_status st = dion_tc(plan, ws, nullptr, 0, 1.0f, stream);
  if (st != MAO_OK) return st;
  // 3. Cholesky QR, twice: Ys -> Ys2 -> Pw (bf16; + the caller's fp32 P)
  const size_t chol_smem = chol_bytes(rank);
  const int nbk = int(ceil_div(rank, 32));
  const unsigned assemble_blocks = unsigned(nbk * (nbk + 1) / 2);
  for (int pass = 0; pass < 2; ++pass) {
    // S = P^T P on the tensor cores from P's parts, assembled in the Cholesky's block layout
    mao_status sg = dion_tc(plan, ws, nullptr, 5, 1.0f, stream, pass);
    if (sg != MAO_OK) return sg;
    profile_before_launch(stream, MAO_PROF_DION_GRAM);
    dion_assemble_kernel<<<dim3(assemble_blocks, nb), 256, 0, stream>>>(c);
    if (!launched()) return MAO_ERR_CUDA;
    profile_before_launch(stream, MAO_PROF_DION_CHOL);
    dion_chol_kernel<<<nb, kCholThreads, chol_smem, stream>>>(c);
    if (!launched()) return MAO_ERR_CUDA;
    // P W^T on the tensor cores: into Ys2 (pass 0), into Pw and the caller's P (pass 1)
    const mao_status st = dion_tc(plan, ws, pass == 1 && P_out ? c.tP : nullptr, 4, 1.0f, stream, pass);
    if (st != MAO_OK) return st;
  }
  // 4. R = B^T P (fp32)
  st = dion_tc(plan, ws, nullptr, 1, 1.0f, stream);
  if (st != MAO_OK) return st;
  // 5. Q = ColumnNormalize(R) (caller's Q), bf16 copies of Q and R
  profile_before_launch(stream, MAO_PROF_DION_NORM);
  dion_norm_kernel<<<dim3(unsigned(plan.ldr / 32), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  profile_before_launch(stream, MAO_PROF_DION_NORM);
  dion_q_kernel<<<dim3(blocks(plan.max_qunits), nb), 256, 0, stream>>>(c);
  if (!launched()) return MAO_ERR_CUDA;
  // 6. M <- B - (1 - mu) P R^T ; X <- X - lr P Q^T (in place)
  // (both in one launch: the X update's table entries follow the M update's)
  return dion_tc(plan, ws, c.tM, 6, -(1.0f - mu), stream, 0, -lr);
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
                     const mao_mat* X_out, float* const* P_out, int32_t batch, int32_t rank,
                     float mu, float lr, int32_t compute, void* workspace,
                     size_t workspace_bytes, void* stream) {
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
    if (X_out) {
      st = check_mat(X_out[b]);
      if (st != MAO_OK) return st;
      if (X_out[b].rows != m || X_out[b].cols != n || X_out[b].dtype != X[b].dtype)
        return MAO_ERR_INVALID_ARG;
      if (X_out[b].data == X[b].data && X_out[b].ld != X[b].ld) return MAO_ERR_INVALID_ARG;
    }
    if (P_out && P_out[b] && reinterpret_cast<uintptr_t>(P_out[b]) % 4 != 0)
      return MAO_ERR_MISALIGNED;
  }
  if (batch > 65535) return MAO_ERR_UNSUPPORTED;
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < dion_workspace_size(X, batch, rank)) return MAO_ERR_WORKSPACE;
  return dion_run(X, M, G, Q, X_out, P_out, batch, rank, mu, lr, workspace,
                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
