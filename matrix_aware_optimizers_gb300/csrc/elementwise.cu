// HBM-bound stages of the optimizer step: momentum, sign + 1-bit pack, majority vote and
// parameter update. All are grouped (one launch covers a batch of matrices of any shapes)
// and move 16 bytes per access where the layout allows it.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mao {
namespace {

constexpr int kEwThreads = 256;
constexpr int kEwUnitsPerThread = 4;  // 8 elements per unit
constexpr int kEwUnitsPerBlock = kEwThreads * kEwUnitsPerThread;
constexpr int kEwMax = 96;            // matrices per launch (kernel-parameter table)

enum EwMode : int32_t { EW_MOMENTUM = 0, EW_UPDATE_U = 1, EW_UPDATE_VOTE = 2 };

struct EwEntry {
  void* a;            // in/out: M (momentum) or W (update)
  const void* b;      // G, U, or packed vote words
  int64_t rows, cols, lda, ldb;
  int64_t units;      // 8-element work units
  int64_t units_per_row;
  int64_t block_begin;
  int32_t dta, dtb;
  int32_t vec;        // 16-byte accesses allowed on a and b
  int32_t flat;       // both contiguous: treated as one row of rows*cols elements
};

struct EwParams {
  EwEntry e[kEwMax];
  int32_t n;
  int32_t mode;
  float scalar;       // mu (momentum) or lr (update)
};

__device__ __forceinline__ int find_entry(const EwParams& p, int64_t block) {
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.e[mid].block_begin <= block) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The per-element arithmetic of each mode, in fp32 with one fused multiply-add.
__device__ __forceinline__ float ew_op(int32_t mode, float s, float a, float b) {
  // momentum: fmaf(mu, m, g); update: fmaf(-lr, d, w)
  return mode == EW_MOMENTUM ? __fmaf_rn(s, a, b) : __fmaf_rn(-s, b, a);
}

__global__ void __launch_bounds__(kEwThreads) ew_kernel(const __grid_constant__ EwParams p) {
  const int ei = find_entry(p, blockIdx.x);
  const EwEntry& e = p.e[ei];
  const int64_t u_begin = (int64_t(blockIdx.x) - e.block_begin) * kEwUnitsPerBlock;
  const uint32_t* vote = reinterpret_cast<const uint32_t*>(e.b);
#pragma unroll 1
  for (int t = 0; t < kEwUnitsPerThread; ++t) {
    const int64_t u = u_begin + t * kEwThreads + threadIdx.x;
    if (u >= e.units) break;
    int64_t row, col0, ncols_row;
    if (e.flat) { row = 0; col0 = u * 8; ncols_row = e.rows * e.cols; }
    else { row = u / e.units_per_row; col0 = (u - row * e.units_per_row) * 8; ncols_row = e.cols; }
    const int valid = int(ncols_row - col0 < 8 ? ncols_row - col0 : 8);
    const int64_t ia = e.flat ? col0 : row * e.lda + col0;
    const int64_t ib = e.flat ? col0 : row * e.ldb + col0;
    const int64_t k0 = e.flat ? col0 : row * e.cols + col0;  // row-major bit index
    float va[8], vb[8];
    if (e.vec && valid == 8) {
      load8(e.a, ia, e.dta, va);
      if (p.mode == EW_UPDATE_VOTE) {
        if ((k0 & 7) == 0) {
          const uint32_t w = vote[k0 >> 5] >> (k0 & 31);
#pragma unroll
          for (int i = 0; i < 8; ++i) vb[i] = ((w >> i) & 1u) ? 1.0f : -1.0f;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int64_t k = k0 + i;
            vb[i] = ((vote[k >> 5] >> (k & 31)) & 1u) ? 1.0f : -1.0f;
          }
        }
      } else {
        load8(e.b, ib, e.dtb, vb);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) va[i] = ew_op(p.mode, p.scalar, va[i], vb[i]);
      store8(e.a, ia, e.dta, va);
    } else {
      for (int i = 0; i < valid; ++i) {
        const float x = load_elem(e.a, ia + i, e.dta);
        float y;
        if (p.mode == EW_UPDATE_VOTE) {
          const int64_t k = k0 + i;
          y = ((vote[k >> 5] >> (k & 31)) & 1u) ? 1.0f : -1.0f;
        } else {
          y = load_elem(e.b, ib + i, e.dtb);
        }
        store_elem(e.a, ia + i, e.dta, ew_op(p.mode, p.scalar, x, y));
      }
    }
  }
}

// Fills one entry of the grouped table; returns its number of blocks.
int64_t make_entry(EwEntry& e, const mao_mat& A, const mao_mat* B, const void* bptr,
                   int32_t dtb, int64_t ldb) {
  e.a = A.data;
  e.b = bptr;
  e.rows = A.rows;
  e.cols = A.cols;
  e.lda = A.ld;
  e.ldb = ldb;
  e.dta = A.dtype;
  e.dtb = dtb;
  const bool contig_a = A.ld == A.cols || A.rows == 1;
  const bool contig_b = B ? (B->ld == B->cols || B->rows == 1) : true;
  e.flat = (contig_a && contig_b) ? 1 : 0;
  bool vec = (reinterpret_cast<uintptr_t>(A.data) % 16 == 0);
  if (B) vec = vec && (reinterpret_cast<uintptr_t>(B->data) % 16 == 0);
  if (!e.flat) {
    vec = vec && (A.cols % 8 == 0) && ((A.ld * elem_size(A.dtype)) % 16 == 0);
    if (B) vec = vec && ((B->ld * elem_size(B->dtype)) % 16 == 0);
  }
  e.vec = vec ? 1 : 0;
  if (e.flat) {
    e.units_per_row = ceil_div(A.rows * A.cols, 8);
    e.units = e.units_per_row;
  } else {
    e.units_per_row = ceil_div(A.cols, 8);
    e.units = e.units_per_row * A.rows;
  }
  return ceil_div(e.units, kEwUnitsPerBlock);
}

mao_status launch_grouped(std::vector<EwEntry>& entries, int32_t mode, float scalar,
                          cudaStream_t stream) {
  size_t pos = 0;
  while (pos < entries.size()) {
    EwParams p;
    p.mode = mode;
    p.scalar = scalar;
    p.n = 0;
    int64_t blocks = 0;
    while (pos < entries.size() && p.n < kEwMax) {
      EwEntry e = entries[pos++];
      if (e.units == 0) continue;
      e.block_begin = blocks;
      blocks += ceil_div(e.units, kEwUnitsPerBlock);
      p.e[p.n++] = e;
    }
    if (p.n == 0) continue;
    if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
    ew_kernel<<<unsigned(blocks), kEwThreads, 0, stream>>>(p);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return MAO_ERR_CUDA;
  }
  return MAO_OK;
}

// ----------------------------------------------------------------- sign + pack

// One thread per 32-bit word: entries k = 32w .. 32w+31 of the row-major matrix.
__global__ void __launch_bounds__(256) sign_pack_kernel(const void* u, int64_t rows, int64_t cols,
                                                        int64_t ld, int32_t dt, int32_t vec,
                                                        uint32_t* bits, int64_t nwords) {
  const int64_t w = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (w >= nwords) return;
  const int64_t k0 = w * 32;
  uint32_t word = 0;
  if (vec) {  // cols % 32 == 0: the word lies inside one row, 16-byte aligned
    const int64_t row = k0 / cols, col0 = k0 - row * cols;
    const int64_t base = row * ld + col0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v[8];
      load8(u, base + 8 * q, dt, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) word |= (v[i] < 0.0f ? 0u : 1u) << (8 * q + i);
    }
  } else {
    const int64_t n = rows * cols;
    for (int i = 0; i < 32; ++i) {
      const int64_t k = k0 + i;
      if (k >= n) break;
      const int64_t row = k / cols, col = k - row * cols;
      const float v = load_elem(u, row * ld + col, dt);
      word |= (v < 0.0f ? 0u : 1u) << i;
    }
  }
  bits[w] = word;
}

// ------------------------------------------------------------------ sign as int8

// One thread per 16 entries k = 16t .. 16t+15 of the row-major matrix: -1 (0xFF) where
// u < 0, else +1. VEC: cols % 16 == 0 and 16-byte aligned rows, one 16-byte store.
template <bool VEC>
__global__ void __launch_bounds__(256) sign_int8_kernel(const void* u, int64_t rows, int64_t cols,
                                                        int64_t ld, int32_t dt, int8_t* s,
                                                        int64_t nchunks) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nchunks) return;
  const int64_t k0 = t * 16;
  if (VEC) {
    const int64_t row = k0 / cols, col0 = k0 - row * cols;
    float v[16];
    load8(u, row * ld + col0, dt, *reinterpret_cast<float(*)[8]>(&v[0]));
    load8(u, row * ld + col0 + 8, dt, *reinterpret_cast<float(*)[8]>(&v[8]));
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) w[q] |= (v[4 * q + i] < 0.0f ? 0xFFu : 0x01u) << (8 * i);
    }
    *reinterpret_cast<uint4*>(s + k0) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    const int64_t n = rows * cols;
    for (int i = 0; i < 16; ++i) {
      const int64_t k = k0 + i;
      if (k >= n) break;
      const int64_t row = k / cols, col = k - row * cols;
      s[k] = load_elem(u, row * ld + col, dt) < 0.0f ? int8_t(-1) : int8_t(1);
    }
  }
}

// ------------------------------------------------------- int8 SUM + threshold vote

// One thread per 32 entries k = 32t .. 32t+31 (one vote word). The W_n int8 signs of each
// entry are summed with per-byte SIMD adds (exact: |sum| <= 127); the sum's sign bit then
// gives S_bar and the vote bit. VEC: 16-byte aligned buffers, all 32 entries in range.
template <bool VEC>
__global__ void __launch_bounds__(256) vote_int8_kernel(const int8_t* __restrict__ s, int32_t nw,
                                                        int64_t stride, int64_t n,
                                                        int8_t* __restrict__ sum,
                                                        int8_t* __restrict__ sbar,
                                                        uint32_t* __restrict__ vote) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t k0 = t * 32;
  if (k0 >= n) return;
  const int valid = n - k0 < 32 ? int(n - k0) : 32;
  uint32_t acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0;
#pragma unroll 4
  for (int m = 0; m < nw; ++m) {
    const int8_t* src = s + int64_t(m) * stride + k0;
    uint32_t x[8];
    if (VEC) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        x[q] = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (4 * q + j < valid) x[q] |= uint32_t(uint8_t(src[4 * q + j])) << (8 * j);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = __vadd4(acc[q], x[q]);
  }
  uint32_t sb[8], word = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t neg = (acc[q] >> 7) & 0x01010101u;  // 1 in each byte whose sum is < 0
    sb[q] = 0x01010101u | (neg * 0xFEu);                // 0x01 (+1) or 0xFF (-1) per byte
    // gather the low bit of each byte of pos into 4 adjacent bits (distinct product terms,
    // no carries): byte i lands on bit 28 + i
    const uint32_t pos = neg ^ 0x01010101u;
    word |= ((pos * 0x10204080u) >> 28) << (4 * q);
  }
  if (valid < 32) word &= (1u << valid) - 1u;
  if (vote) vote[t] = word;
  if (VEC) {
    if (sum) {
      uint4* d = reinterpret_cast<uint4*>(sum + k0);
      d[0] = make_uint4(acc[0], acc[1], acc[2], acc[3]);
      d[1] = make_uint4(acc[4], acc[5], acc[6], acc[7]);
    }
    if (sbar) {
      uint4* d = reinterpret_cast<uint4*>(sbar + k0);
      d[0] = make_uint4(sb[0], sb[1], sb[2], sb[3]);
      d[1] = make_uint4(sb[4], sb[5], sb[6], sb[7]);
    }
  } else {
    for (int j = 0; j < valid; ++j) {
      if (sum) sum[k0 + j] = int8_t(uint8_t(acc[j >> 2] >> (8 * (j & 3))));
      if (sbar) sbar[k0 + j] = int8_t(uint8_t(sb[j >> 2] >> (8 * (j & 3))));
    }
  }
}

// --------------------------------------------------------------- majority vote

constexpr int kMaxPlanes = 16;  // counts up to 65535 workers

// Adds one 32-lane word of bits into a bit-sliced binary counter (plane p holds bit p of
// every lane's count): a ripple of half adders, three logic ops per plane. PL planes are
// held in registers (PL >= P, the planes the worker count needs).
template <int PL>
__device__ __forceinline__ void counter_add(uint32_t (&plane)[PL], int P, uint32_t x) {
  uint32_t carry = x;
#pragma unroll
  for (int p = 0; p < PL; ++p) {
    if (p < P) {
      const uint32_t t = plane[p] & carry;
      plane[p] ^= carry;
      carry = t;
    }
  }
}

// Lanes whose count is >= T, by comparing the bit-sliced count with T from the top bit.
template <int PL>
__device__ __forceinline__ uint32_t counter_ge(const uint32_t (&plane)[PL], int P, uint32_t T) {
  uint32_t gt = 0, eq = 0xFFFFFFFFu;
#pragma unroll
  for (int p = PL - 1; p >= 0; --p) {
    if (p < P) {
      if ((T >> p) & 1u) {
        eq &= plane[p];
      } else {
        gt |= eq & plane[p];
        eq &= ~plane[p];
      }
    }
  }
  return gt | eq;
}

template <int V, int PL>
__global__ void __launch_bounds__(256) vote_kernel(const uint32_t* __restrict__ bits, int32_t nw,
                                                   int64_t stride, int64_t nwords, int64_t nbits,
                                                   int64_t total_words, uint32_t* __restrict__ vote,
                                                   int P, uint32_t T) {
  const int64_t w0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * V;
  if (w0 >= nwords) return;
  uint32_t plane[V][PL];
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int p = 0; p < PL; ++p) plane[v][p] = 0;
  // unrolled so that several workers' loads are in flight before the counter updates
#pragma unroll 4
  for (int m = 0; m < nw; ++m) {
    const uint32_t* src = bits + int64_t(m) * stride + w0;
    if (V == 4) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(src));
      counter_add<PL>(plane[0], P, x.x);
      counter_add<PL>(plane[V > 1 ? 1 : 0], P, x.y);
      counter_add<PL>(plane[V > 2 ? 2 : 0], P, x.z);
      counter_add<PL>(plane[V > 3 ? 3 : 0], P, x.w);
    } else {
      counter_add<PL>(plane[0], P, __ldg(src));
    }
  }
  uint32_t out[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    out[v] = counter_ge<PL>(plane[v], P, T);
    const int64_t w = w0 + v;
    if (w == total_words - 1 && (nbits & 31)) out[v] &= (1u << (nbits & 31)) - 1u;
  }
  if (V == 4) {
    *reinterpret_cast<uint4*>(vote + w0) = make_uint4(out[0], out[V > 1 ? 1 : 0],
                                                      out[V > 2 ? 2 : 0], out[V > 3 ? 3 : 0]);
  } else {
    vote[w0] = out[0];
  }
}

template <int V>
void launch_vote(int64_t blocks, cudaStream_t stream, const uint32_t* bits, int32_t nw,
                 int64_t stride, int64_t nwords, int64_t nbits, int64_t total_words,
                 uint32_t* vote, int P, uint32_t T) {
  if (P <= 4)
    vote_kernel<V, 4><<<unsigned(blocks), 256, 0, stream>>>(bits, nw, stride, nwords, nbits,
                                                            total_words, vote, P, T);
  else if (P <= 8)
    vote_kernel<V, 8><<<unsigned(blocks), 256, 0, stream>>>(bits, nw, stride, nwords, nbits,
                                                            total_words, vote, P, T);
  else
    vote_kernel<V, kMaxPlanes><<<unsigned(blocks), 256, 0, stream>>>(bits, nw, stride, nwords,
                                                                     nbits, total_words, vote,
                                                                     P, T);
}

// The vote and the update of W in one pass: thread w forms vote word w (as vote_kernel, one
// word per thread) and applies it to W's entries k = 32 w .. 32 w + 31 (row-major),
// W <- fma(-lr, v, W) with v = +1 / -1, rounded to W's dtype (the update kernel's
// arithmetic). With vec (contiguous 16-byte-aligned rows, cols a multiple of 8) the 32
// entries are four 8-element units of one row.
template <int PL>
__global__ void __launch_bounds__(256) vote_update_kernel(const uint32_t* __restrict__ bits, int32_t nw,
                                                          int64_t stride, int64_t nbits,
                                                          uint32_t* __restrict__ vote, int P, uint32_t T,
                                                          void* W, int64_t cols, int64_t ld, int32_t dt,
                                                          int32_t vec, float lr) {
  const int64_t nwords = (nbits + 31) / 32;
  const int64_t w = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (w >= nwords) return;
  uint32_t plane[PL];
#pragma unroll
  for (int p = 0; p < PL; ++p) plane[p] = 0;
#pragma unroll 4
  for (int m = 0; m < nw; ++m) counter_add<PL>(plane, P, __ldg(bits + int64_t(m) * stride + w));
  uint32_t v = counter_ge<PL>(plane, P, T);
  if (w == nwords - 1 && (nbits & 31)) v &= (1u << (nbits & 31)) - 1u;
  vote[w] = v;
  const int64_t k0 = 32 * w;
  const int cnt = int(nbits - k0 < 32 ? nbits - k0 : 32);
  const int64_t row0 = k0 / cols, col0 = k0 - row0 * cols;
  if (vec && cnt == 32 && col0 + 32 <= cols) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float a[8];
      const int64_t at = row0 * ld + col0 + 8 * u;
      load8(W, at, dt, a);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = __fmaf_rn(-lr, ((v >> (8 * u + i)) & 1u) ? 1.0f : -1.0f, a[i]);
      store8(W, at, dt, a);
    }
  } else {
    for (int b = 0; b < cnt; ++b) {
      const int64_t k = k0 + b, row = k / cols, col = k - row * cols;
      const float x = load_elem(W, row * ld + col, dt);
      store_elem(W, row * ld + col, dt, __fmaf_rn(-lr, ((v >> b) & 1u) ? 1.0f : -1.0f, x));
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- entry points

mao_status momentum_launch(const mao_mat* M, const mao_mat* G, int32_t batch, float mu,
                           cudaStream_t stream) {
  std::vector<EwEntry> entries(batch);
  for (int i = 0; i < batch; ++i) make_entry(entries[i], M[i], &G[i], G[i].data, G[i].dtype, G[i].ld);
  return launch_grouped(entries, EW_MOMENTUM, mu, stream);
}

mao_status update_launch(const mao_mat* W, const uint32_t* const* vote, const mao_mat* U,
                         int32_t batch, float lr, cudaStream_t stream) {
  std::vector<EwEntry> entries(batch);
  for (int i = 0; i < batch; ++i) {
    if (vote) make_entry(entries[i], W[i], nullptr, vote[i], MAO_F32, W[i].cols);
    else make_entry(entries[i], W[i], &U[i], U[i].data, U[i].dtype, U[i].ld);
  }
  return launch_grouped(entries, vote ? EW_UPDATE_VOTE : EW_UPDATE_U, lr, stream);
}

mao_status sign_pack_launch(const mao_mat& U, uint32_t* bits, cudaStream_t stream) {
  const int64_t n = U.rows * U.cols;
  const int64_t nwords = ceil_div(n, 32);
  const bool vec = (U.cols % 32 == 0) && vec8_ok(U);
  const int64_t blocks = ceil_div(nwords, 256);
  if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
  sign_pack_kernel<<<unsigned(blocks), 256, 0, stream>>>(U.data, U.rows, U.cols, U.ld, U.dtype,
                                                         vec ? 1 : 0, bits, nwords);
  count_launch();
  return cuda_status(cudaGetLastError());
}

mao_status sign_int8_launch(const mao_mat& U, int8_t* s, cudaStream_t stream) {
  const int64_t n = U.rows * U.cols;
  const int64_t nchunks = ceil_div(n, 16);
  const bool vec = (U.cols % 16 == 0) && vec8_ok(U) && (reinterpret_cast<uintptr_t>(s) % 16 == 0);
  const int64_t blocks = ceil_div(nchunks, 256);
  if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
  if (vec)
    sign_int8_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(U.data, U.rows, U.cols, U.ld,
                                                                 U.dtype, s, nchunks);
  else
    sign_int8_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(U.data, U.rows, U.cols, U.ld,
                                                                  U.dtype, s, nchunks);
  count_launch();
  return cuda_status(cudaGetLastError());
}

mao_status vote_int8_launch(const int8_t* s, int32_t n_workers, int64_t stride, int64_t n,
                            int8_t* sum, int8_t* sbar, uint32_t* vote, cudaStream_t stream) {
  auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  // 16-byte path over the first floor(n/32)*32 entries, byte path for the rest
  const bool vec = a16(s) && stride % 16 == 0 && (!sum || a16(sum)) && (!sbar || a16(sbar));
  const int64_t bulk = vec ? (n / 32) * 32 : 0;
  if (bulk > 0) {
    const int64_t blocks = ceil_div(bulk / 32, 256);
    if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
    vote_int8_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(s, n_workers, stride, bulk, sum,
                                                                 sbar, vote);
    count_launch();
  }
  if (n > bulk) {
    const int64_t blocks = ceil_div(ceil_div(n - bulk, 32), 256);
    if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
    vote_int8_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(
        s + bulk, n_workers, stride, n - bulk, sum ? sum + bulk : nullptr,
        sbar ? sbar + bulk : nullptr, vote ? vote + bulk / 32 : nullptr);
    count_launch();
  }
  return cuda_status(cudaGetLastError());
}

mao_status vote_update_launch(const uint32_t* bits, int32_t n_workers, int64_t stride,
                              int64_t nbits, uint32_t* vote, const mao_mat& W, float lr,
                              cudaStream_t stream) {
  const int64_t nwords = ceil_div(nbits, 32);
  int P = 0;
  while ((int64_t(1) << P) <= n_workers) ++P;  // n_workers < 2^P
  const uint32_t T = uint32_t((n_workers + 1) / 2);  // count of +1 needed: 2*cnt >= W_n
  const bool vec = W.cols % 8 == 0 && reinterpret_cast<uintptr_t>(W.data) % 16 == 0 &&
                   (W.ld * elem_size(W.dtype)) % 16 == 0;
  const int64_t blocks = ceil_div(nwords, 256);
  if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
  if (P <= 4)
    vote_update_kernel<4><<<unsigned(blocks), 256, 0, stream>>>(bits, n_workers, stride, nbits, vote, P, T,
                                                                W.data, W.cols, W.ld, W.dtype, vec, lr);
  else if (P <= 8)
    vote_update_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(bits, n_workers, stride, nbits, vote, P, T,
                                                                W.data, W.cols, W.ld, W.dtype, vec, lr);
  else
    vote_update_kernel<kMaxPlanes><<<unsigned(blocks), 256, 0, stream>>>(
        bits, n_workers, stride, nbits, vote, P, T, W.data, W.cols, W.ld, W.dtype, vec, lr);
  count_launch();
  return cuda_status(cudaGetLastError());
}

mao_status vote_launch(const uint32_t* bits, int32_t n_workers, int64_t stride, int64_t nbits,
                       uint32_t* vote, cudaStream_t stream) {
  const int64_t nwords = ceil_div(nbits, 32);
  int P = 0;
  while ((int64_t(1) << P) <= n_workers) ++P;  // n_workers < 2^P
  const uint32_t T = uint32_t((n_workers + 1) / 2);  // count of +1 needed: 2*cnt >= W_n
  // 16-byte path over the first floor(nwords/4)*4 words, one word per thread for the rest
  const bool v4 = (stride % 4 == 0) && (reinterpret_cast<uintptr_t>(bits) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(vote) % 16 == 0);
  const int64_t bulk = v4 ? (nwords / 4) * 4 : 0;
  if (bulk > 0) {
    const int64_t blocks = ceil_div(bulk / 4, 256);
    launch_vote<4>(blocks, stream, bits, n_workers, stride, bulk, nbits, nwords, vote, P, T);
    count_launch();
  }
  if (nwords > bulk) {
    const int64_t rest = nwords - bulk;
    const int64_t blocks = ceil_div(rest, 256);
    launch_vote<1>(blocks, stream, bits + bulk, n_workers, stride, rest, nbits - bulk * 32,
                   nwords - bulk, vote + bulk, P, T);
    count_launch();
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace mao
