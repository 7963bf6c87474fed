// Newton–Schulz orchestration: shape grouping, workspace layout, staging with the
// Frobenius norm, the per-iteration chain of three grouped products, and the fp32 FFMA
// product kernel of the accuracy path.
//
// Per iteration ("分散ニュートン・シュルツ" of the Megatron Muon article counts three matrix
// products per Newton–Schulz iteration; its "SYRK" section maps the first two onto
// symmetric rank-k updates that still produce the full matrix):
//   A = X X^T ; B = b A + c A A ; X <- a X + B X
// evaluated as X <- (a I + B) X, with a I added on the diagonal by the second product.
// The first iteration reads the staged, unnormalised input and applies s = 1/(||X||_F+eps)
// as s^2 in the first product's epilogue and s in the third's, so the normalisation costs
// no pass of its own.
#include <algorithm>
#include <cmath>
#include <map>
#include <utility>

#include "common.cuh"
#include "ns_plan.h"
#include "ns_small.h"

namespace mao {

// ------------------------------------------------------------------- planning

bool make_ns_plan(const mao_mat* X, int32_t batch, int32_t compute, NsPlan& plan) {
  plan = NsPlan();
  plan.es = compute == MAO_BF16 ? 2 : 4;
  std::map<std::pair<int64_t, int64_t>, int> gid;
  std::vector<std::vector<int>> members;
  for (int b = 0; b < batch; ++b) {
    const auto key = std::make_pair(X[b].rows, X[b].cols);
    auto it = gid.find(key);
    if (it == gid.end()) {
      gid.emplace(key, int(members.size()));
      members.emplace_back();
      members.back().push_back(b);
    } else {
      members[it->second].push_back(b);
    }
  }
  // groups in decreasing per-matrix work (4 m^2 n + 2 m^3), ties in order of appearance
  std::vector<int> order(members.size());
  for (size_t g = 0; g < order.size(); ++g) order[g] = int(g);
  auto work = [&](int g) {
    const double R = double(X[members[g][0]].rows), C = double(X[members[g][0]].cols);
    const double m = std::min(R, C), n = std::max(R, C);
    return 4.0 * m * m * n + 2.0 * m * m * m;
  };
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return work(x) > work(y); });

  plan.slot_of.assign(batch, -1);
  plan.partial_begin.assign(batch + 1, 0);
  int slot = 0;
  for (int g : order) {
    NsGroupPlan gp;
    gp.R = X[members[g][0]].rows;
    gp.C = X[members[g][0]].cols;
    gp.m = std::min(gp.R, gp.C);
    gp.n = std::max(gp.R, gp.C);
    gp.tall = gp.R > gp.C;
    gp.count = int32_t(members[g].size());
    gp.slot0 = slot;
    gp.ldx = round_up(gp.C, tc::LD_ALIGN);
    gp.lda = round_up(gp.m, tc::LD_ALIGN);
    for (int b : members[g]) {
      plan.slot_of[b] = slot;
      plan.input_of.push_back(b);
      ++slot;
    }
    plan.groups.push_back(gp);
  }
  int64_t np = 0;
  for (const auto& gp : plan.groups) {
    for (int j = 0; j < gp.count; ++j) {
      plan.partial_begin[gp.slot0 + j] = np;
      np += ceil_div(gp.R * (gp.ldx / 8), kStageUnitsPerBlock);
    }
  }
  plan.partial_begin[batch] = np;
  plan.n_partials = np;

  size_t off = 0;
  plan.off_out_table = off;
  off = size_t(round_up(int64_t(off + sizeof(OutEntry) * batch), 256));
  plan.off_scale = off;
  off = size_t(round_up(int64_t(off + sizeof(float) * batch), 256));
  plan.off_prange = off;
  off = size_t(round_up(int64_t(off + 2 * sizeof(int64_t) * batch), 256));
  plan.off_partials = off;
  off = size_t(round_up(int64_t(off + sizeof(float) * np), 1024));
  for (auto& gp : plan.groups) {
    const size_t xb = size_t(gp.count) * size_t(gp.R) * size_t(gp.ldx) * plan.es;
    const size_t ab = size_t(gp.count) * size_t(gp.m) * size_t(gp.lda) * plan.es;
    gp.off_x[0] = off;
    off = size_t(round_up(int64_t(off + xb), 1024));
    gp.off_x[1] = off;
    off = size_t(round_up(int64_t(off + xb), 1024));
    gp.off_a = off;
    off = size_t(round_up(int64_t(off + ab), 1024));
    gp.off_b = off;
    off = size_t(round_up(int64_t(off + ab), 1024));
  }
  plan.total = off;
  return true;
}

size_t ns_workspace_size(const mao_mat* X, int32_t batch, int32_t compute) {
  NsPlan plan;
  make_ns_plan(X, batch, compute, plan);
  return plan.total;
}

namespace {

// ------------------------------------------------------------ stage-in + norm

constexpr int kStageMax = 48;

struct StageEntry {
  const void* src;
  void* dst;
  const void* g;        // momentum fused in (muon_step): G, and src is written back
  int64_t src_ld, dst_ld, rows, cols, units_per_row, units;
  int64_t g_ld;
  int64_t block_begin;  // first block of this entry in the launch
  int64_t partial0;     // partial-sum index of that block
  int64_t nblocks;      // blocks (= partial sums) of this entry
  OutEntry out;
  int32_t src_dt, vec_src, slot, g_dt;
};

struct StageParams {
  StageEntry e[kStageMax];
  int32_t n, ws_dt;
  float mu;             // momentum coefficient of the fused entries
  OutEntry* table;
  int64_t* prange;      // per slot: first partial, number of partials
  float* partials;
};

// Loads the `valid` (<= 8) source elements (row, col0 .. col0+valid-1) of a staged input as
// fp32, zeros beyond. f32/bf16 take 16-byte loads when `vec`; int8 takes one 8-byte load when
// `vec`; packed signs read the (at most two) words holding the 8 bits.
__device__ __forceinline__ void stage_load8(const StageEntry& e, int64_t row, int64_t col0,
                                            int valid, float (&v)[8]) {
  if (e.src_dt == MAO_SIGN1) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(e.src);
    const int64_t k = row * e.cols + col0;
    const int64_t wi = k >> 5;
    const int sh = int(k & 31);
    uint64_t x = w[wi];
    if (sh + valid > 32) x |= uint64_t(w[wi + 1]) << 32;
    x >>= sh;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = i < valid ? (((x >> i) & 1u) ? 1.0f : -1.0f) : 0.0f;
    return;
  }
  if (e.src_dt == MAO_I8) {
    const int8_t* p = reinterpret_cast<const int8_t*>(e.src) + row * e.src_ld + col0;
    if (e.vec_src && valid == 8) {
      const uint2 raw = *reinterpret_cast<const uint2*>(p);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] = float(int8_t(raw.x >> (8 * i)));
        v[4 + i] = float(int8_t(raw.y >> (8 * i)));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = i < valid ? float(p[i]) : 0.0f;
    }
    return;
  }
  if (e.vec_src && valid == 8) {
    load8(e.src, row * e.src_ld + col0, e.src_dt, v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = i < valid ? load_elem(e.src, row * e.src_ld + col0 + i, e.src_dt) : 0.0f;
  }
}

// One unit (8 elements of a row, `valid` of them inside the matrix) of the general path:
// the source values as fp32. With momentum fused in, M <- fmaf(mu, M, G) rounded to M's
// dtype is written back, and the rounded values are what Newton–Schulz orthogonalises (as
// if M had been updated first).
__device__ __forceinline__ void stage_unit(const StageEntry& e, float mu, int64_t row,
                                           int64_t col0, int valid, float (&v)[8]) {
  stage_load8(e, row, col0, valid, v);
  if (!e.g || valid <= 0) return;
  float gv[8];
  if (e.vec_src && valid == 8) {
    load8(e.g, row * e.g_ld + col0, e.g_dt, gv);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) gv[i] = i < valid ? load_elem(e.g, row * e.g_ld + col0 + i, e.g_dt) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float m = __fmaf_rn(mu, v[i], gv[i]);
    v[i] = i < valid ? (e.src_dt == MAO_BF16 ? __bfloat162float(__float2bfloat16_rn(m)) : m) : 0.0f;
  }
  void* mo = const_cast<void*>(e.src);
  if (e.vec_src && valid == 8) {
    store8(mo, row * e.src_ld + col0, e.src_dt, v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < valid) store_elem(mo, row * e.src_ld + col0 + i, e.src_dt, v[i]);
  }
}

// Copies each input into its workspace slot (converting to the compute type) and writes
// one fp32 partial sum of squares per block; records the slot's output entry.
__global__ void __launch_bounds__(kStageThreads) stage_in_kernel(const __grid_constant__ StageParams p) {
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.e[mid].block_begin <= int64_t(blockIdx.x)) lo = mid; else hi = mid - 1;
  }
  const StageEntry& e = p.e[lo];
  const int64_t blk = int64_t(blockIdx.x) - e.block_begin;
  if (blk == 0 && threadIdx.x == 0) {
    p.table[e.slot] = e.out;
    p.prange[2 * e.slot] = e.partial0;
    p.prange[2 * e.slot + 1] = e.nblocks;
  }
  float sq = 0.0f;
  const int64_t u0 = blk * kStageUnitsPerBlock;
  constexpr int U = kStageUnitsPerBlock / kStageThreads;
  if (e.src_dt == MAO_BF16 && p.ws_dt == MAO_BF16 && e.vec_src && (!e.g || e.g_dt == MAO_BF16) &&
      e.units <= 0xFFFFFFFFll) {
    // bf16 rows with 16-byte accesses: every unit's loads are issued before any arithmetic,
    // and the values stay packed until used. Same arithmetic and order as the loop below.
    const uint32_t upr = uint32_t(e.units_per_row);
    uint4 m[U], g[U];
    uint32_t row[U], col0[U];
    bool live[U], full[U];
#pragma unroll
    for (int t = 0; t < U; ++t) {
      const int64_t u = u0 + t * kStageThreads + threadIdx.x;
      live[t] = u < e.units;
      const uint32_t uu = live[t] ? uint32_t(u) : 0u;
      row[t] = uu / upr;
      col0[t] = (uu - row[t] * upr) * 8u;
      full[t] = live[t] && int64_t(col0[t]) + 8 <= e.cols;
      if (full[t]) {
        m[t] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(e.src) +
                                               int64_t(row[t]) * e.src_ld + col0[t]);
        if (e.g)
          g[t] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(e.g) +
                                                      int64_t(row[t]) * e.g_ld + col0[t]));
      }
    }
#pragma unroll
    for (int t = 0; t < U; ++t) {
      if (!live[t]) continue;
      float v[8];
      if (full[t]) {
        uint32_t* h = reinterpret_cast<uint32_t*>(&m[t]);
        const uint32_t* hg = reinterpret_cast<const uint32_t*>(&g[t]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[2 * k] = __uint_as_float(h[k] << 16);
          v[2 * k + 1] = __uint_as_float(h[k] & 0xFFFF0000u);
        }
        if (e.g) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(
                __fmaf_rn(p.mu, v[2 * k], __uint_as_float(hg[k] << 16)),
                __fmaf_rn(p.mu, v[2 * k + 1], __uint_as_float(hg[k] & 0xFFFF0000u)));
            h[k] = *reinterpret_cast<const uint32_t*>(&b);
            v[2 * k] = __uint_as_float(h[k] << 16);
            v[2 * k + 1] = __uint_as_float(h[k] & 0xFFFF0000u);
          }
          *reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(
              reinterpret_cast<const __nv_bfloat16*>(e.src) + int64_t(row[t]) * e.src_ld + col0[t])) = m[t];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sq = __fmaf_rn(v[i], v[i], sq);
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(e.dst) + int64_t(row[t]) * e.dst_ld +
                                  col0[t]) = m[t];
      } else {
        const int64_t left = e.cols - int64_t(col0[t]);
        const int valid = int(left >= 8 ? 8 : (left > 0 ? left : 0));
        stage_unit(e, p.mu, row[t], col0[t], valid, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) sq = __fmaf_rn(v[i], v[i], sq);
        store8(e.dst, int64_t(row[t]) * e.dst_ld + col0[t], p.ws_dt, v);
      }
    }
  } else {
#pragma unroll 1
    for (int t = 0; t < U; ++t) {
      const int64_t u = u0 + t * kStageThreads + threadIdx.x;
      if (u >= e.units) break;
      // units cover the padded workspace row: columns >= cols are written as zeros
      const int64_t row = u / e.units_per_row;
      const int64_t col0 = (u - row * e.units_per_row) * 8;
      const int64_t left = e.cols - col0;
      const int valid = int(left >= 8 ? 8 : (left > 0 ? left : 0));
      float v[8];
      stage_unit(e, p.mu, row, col0, valid, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) sq = __fmaf_rn(v[i], v[i], sq);
      store8(e.dst, row * e.dst_ld + col0, p.ws_dt, v);
    }
  }
  // fixed-order block reduction: warp tree, then warp 0 over the warp sums
  __shared__ float wsum[kStageThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x < 32) {
    float x = threadIdx.x < kStageThreads / 32 ? wsum[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    if (threadIdx.x == 0) p.partials[e.partial0 + blk] = x;
  }
}

// One warp per slot: fp64 sum of the slot's partials in a fixed order, then
// s = 1 / (sqrt(sum) + eps).
__global__ void __launch_bounds__(32) finalize_scale_kernel(const float* partials,
                                                            const int64_t* prange, float* scale,
                                                            float eps) {
  const int slot = blockIdx.x;
  const int64_t b0 = prange[2 * slot], nb = prange[2 * slot + 1];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < nb; i += 32) acc += double(partials[b0 + i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (threadIdx.x == 0) scale[slot] = float(1.0 / (sqrt(acc) + double(eps)));
}

// ------------------------------------------------------- fp32 FFMA product path

constexpr int kSimtMaxGroups = 8;
constexpr int kSimtTile = 128;
constexpr int kSimtK = 8;

struct SimtGroup {
  const float* a;
  const float* b;
  float* out;
  const float* res;
  int64_t a_ms, a_si, a_sk;     // operand A(i, k) = a[z*a_ms + i*a_si + k*a_sk]
  int64_t b_ms, b_sj, b_sk;     // operand B(j, k) = b[z*b_ms + j*b_sj + k*b_sk]
  int64_t out_ms, out_ld, res_ms, res_ld;
  int64_t block_begin;
  int32_t M, N, K, count, slot0, syrk, tiles_m, tiles_n, final_out, orig_cols;
};

struct SimtParams {
  SimtGroup g[kSimtMaxGroups];
  int32_t ngroups, stage;
  float a, b, c;
  const float* scale;
  const OutEntry* out_table;
};

// One operand's slice of a k-step: kSimtTile rows (i) x kSimtK columns (k) of
// src(i, k) = src[i*si + k*sk], four elements per thread. When k is the contiguous index
// (sk == 1) eight neighbouring threads read eight consecutive k of one row, otherwise 128
// neighbouring threads read 128 consecutive rows of one k, so the loads coalesce either
// way. Outside [0, rows) x [0, K) the values are zero.
struct SimtSlice {
  float v[4];
};
__device__ __forceinline__ void simt_load(SimtSlice& t, const float* src, int64_t si, int64_t sk,
                                          int r0, int rows, int k0, int K) {
  const bool kfast = sk == 1;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x + 256 * q;
    const int ii = kfast ? e >> 3 : e & (kSimtTile - 1);
    const int kk = kfast ? e & 7 : e >> 7;
    const int gi = r0 + ii, gk = k0 + kk;
    t.v[q] = (gi < rows && gk < K) ? src[int64_t(gi) * si + int64_t(gk) * sk] : 0.0f;
  }
}
__device__ __forceinline__ void simt_store(const SimtSlice& t, float (*S)[kSimtTile + 4], bool kfast) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x + 256 * q;
    const int ii = kfast ? e >> 3 : e & (kSimtTile - 1);
    const int kk = kfast ? e & 7 : e >> 7;
    S[kk][ii] = t.v[q];
  }
}

// D(i, j) = sum_k A(i, k) B(j, k) on a 128 x 128 tile, fp32 FFMA: thread (ty, tx) of 16 x 16
// holds rows ty*4 + {0..3} and 64 + ty*4 + {0..3}, columns tx*4 + {0..3} and
// 64 + tx*4 + {0..3} (conflict-free 16-byte shared-memory reads); the next k-step's slices
// are loaded into registers while the current one is multiplied.
__global__ void __launch_bounds__(256) ns_simt_kernel(const __grid_constant__ SimtParams p) {
  int gi = 0;
  while (gi + 1 < p.ngroups && p.g[gi + 1].block_begin <= int64_t(blockIdx.x)) ++gi;
  const SimtGroup& G = p.g[gi];
  const int64_t local = int64_t(blockIdx.x) - G.block_begin;
  const int tiles = G.tiles_m * G.tiles_n;
  const int z = int(local / tiles);
  const int r = int(local - int64_t(z) * tiles);
  const int tm = r / G.tiles_n, tn = r - tm * G.tiles_n;
  if (G.syrk && tm > tn) return;  // lower tiles come from the mirror of upper ones
  const int row0 = tm * kSimtTile, col0 = tn * kSimtTile;
  const float* A = G.a + int64_t(z) * G.a_ms;
  const float* B = G.b + int64_t(z) * G.b_ms;

  __shared__ __align__(16) float As[kSimtK][kSimtTile + 4];
  __shared__ __align__(16) float Bs[kSimtK][kSimtTile + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  SimtSlice ta, tb;
  simt_load(ta, A, G.a_si, G.a_sk, row0, G.M, 0, G.K);
  simt_load(tb, B, G.b_sj, G.b_sk, col0, G.N, 0, G.K);
  for (int k0 = 0; k0 < G.K; k0 += kSimtK) {
    simt_store(ta, As, G.a_sk == 1);
    simt_store(tb, Bs, G.b_sk == 1);
    __syncthreads();
    if (k0 + kSimtK < G.K) {
      simt_load(ta, A, G.a_si, G.a_sk, row0, G.M, k0 + kSimtK, G.K);
      simt_load(tb, B, G.b_sj, G.b_sk, col0, G.N, k0 + kSimtK, G.K);
    }
#pragma unroll
    for (int kk = 0; kk < kSimtK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

  const int slot = G.slot0 + z;
  const float s = p.scale ? p.scale[slot] : 1.0f;
  float* out = G.out + int64_t(z) * G.out_ms;
  const float* res = G.res + int64_t(z) * G.res_ms;
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = row0 + (ii < 4 ? ty * 4 + ii : 64 + ty * 4 + ii - 4);
    if (i >= G.M) continue;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = col0 + (jj < 4 ? tx * 4 + jj : 64 + tx * 4 + jj - 4);
      if (j >= G.N) continue;
      const float v = acc[ii][jj];
      if (p.stage == NS_GRAM || p.stage == NS_POLY) {
        if (j < i) continue;
        const float w = p.stage == NS_GRAM
                            ? (s * s) * v
                            : __fmaf_rn(p.c, v, p.b * res[int64_t(i) * G.res_ld + j]) + (i == j ? p.a : 0.0f);
        out[int64_t(i) * G.out_ld + j] = w;
        if (j > i) out[int64_t(j) * G.out_ld + i] = w;
      } else {
        const float w = s * v;
        if (G.final_out) {
          const OutEntry& e = p.out_table[slot];
          if (e.out) store_elem(e.out, int64_t(i) * e.ld + j, e.dtype, w);
          if (e.bits && !(w < 0.0f)) {
            const int64_t k = int64_t(i) * G.orig_cols + j;
            atomicOr(e.bits + (k >> 5), 1u << (k & 31));
          }
        } else {
          out[int64_t(i) * G.out_ld + j] = w;
        }
      }
    }
  }
}

// ------------------------------------------------------------------- driver

struct Buffers {
  uint8_t* ws;
  const NsPlan* plan;
  void* x(const NsGroupPlan& g, int which) const { return ws + g.off_x[which]; }
  void* a(const NsGroupPlan& g) const { return ws + g.off_a; }
  void* b(const NsGroupPlan& g) const { return ws + g.off_b; }
};

int syrk_tiles(int64_t m) {
  int t = 0;
  for (int64_t ib = 0; tc::TILE_M * ib < m; ++ib) t += int(ceil_div(m - tc::TILE_M * ib, tc::BN));
  return t;
}

// update_alpha (finite): the last product updates the outputs in place,
// out <- out + update_alpha * U (TC_UPDATE), instead of writing U.
mao_status run_tc_stage(const Buffers& buf, const std::vector<const NsGroupPlan*>& round,
                        int stage, int cur, bool first, bool last, const float* co,
                        const float* scale, const OutEntry* table, int out_mode,
                        cudaStream_t stream, float update_alpha = NAN) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.out_mode = last ? out_mode : tc::OUT_WORKSPACE;
  p.ngroups = int32_t(round.size());
  p.stage = stage;
  p.a = co[0];
  p.b = co[1];
  p.c = co[2];
  p.scale = first ? scale : nullptr;
  p.out_table = table;
  p.timeout_ns = wait_limit_ns();
  int tiles = 0;
  for (size_t gi = 0; gi < round.size(); ++gi) {
    const NsGroupPlan& g = *round[gi];
    TcGroup& G = p.g[gi];
    G.count = g.count;
    G.slot0 = g.slot0;
    G.orig_cols = int32_t(g.C);
    const void* X = buf.x(g, cur);
    const int64_t xs = g.R * g.ldx, as = g.m * g.lda;
    mao_status st = MAO_OK;
    const void *srcA, *srcB;
    int64_t rowsA, ldA, rowsB, ldB;
    if (stage == NS_GRAM) {
      srcA = srcB = X;
      rowsA = rowsB = g.R;
      ldA = ldB = g.ldx;
      G.a_mn = G.b_mn = g.tall ? 1 : 0;
      G.M = G.N = int32_t(g.m);
      G.K = int32_t(g.n);
      G.out = buf.a(g);
      G.out_ld = g.lda;
      G.out_mstride = as;
      G.res = nullptr;
      G.syrk = 1;
      G.same_ab = 1;
    } else if (stage == NS_POLY) {
      srcA = srcB = buf.a(g);
      rowsA = rowsB = g.m;
      ldA = ldB = g.lda;
      G.a_mn = G.b_mn = 0;
      G.a_sym = G.b_sym = 1;
      G.M = G.N = G.K = int32_t(g.m);
      G.out = buf.b(g);
      G.out_ld = g.lda;
      G.out_mstride = as;
      G.res = buf.a(g);
      G.res_ld = g.lda;
      G.res_mstride = as;
      G.syrk = 1;
      G.same_ab = 1;
    } else {
      if (!g.tall) {  // X' = B' X : A-operand B' (K-major), B-operand X (MN-major)
        srcA = buf.b(g); rowsA = g.m; ldA = g.lda;
        srcB = X; rowsB = g.R; ldB = g.ldx;
        G.a_mn = 0;
        G.b_mn = 1;
        G.a_sym = 1;
      } else {        // X' = X B' : A-operand X (K-major), B-operand B' (K-major)
        srcA = X; rowsA = g.R; ldA = g.ldx;
        srcB = buf.b(g); rowsB = g.m; ldB = g.lda;
        G.a_mn = 0;
        G.b_mn = 0;
        G.b_sym = 1;
      }
      G.M = int32_t(g.R);
      G.N = int32_t(g.C);
      G.K = int32_t(g.m);
      G.out = last ? nullptr : buf.x(g, 1 - cur);
      G.out_ld = g.ldx;
      G.out_mstride = xs;
      G.res = nullptr;
      G.syrk = 0;
      G.final_out = last ? 1 : 0;
    }
    // One 4-D map per buffer serves both operand orientations: box = 64 columns x 128 rows
    // x 2 column chunks; K-major operands step the chunk along K, MN-major ones along M/N.
    st = tc_encode_map(&G.tmA, srcA, rowsA, ldA, g.count);
    if (st == MAO_OK) st = tc_encode_map(&G.tmB, srcB, rowsB, ldB, g.count);
    if (st == MAO_OK && G.out)
      st = tc_encode_store_map(&G.tmOR, G.out, G.M, G.out_ld, g.count);
    if (st != MAO_OK) return st;
    G.tiles_m = int32_t(ceil_div(G.M, tc::TILE_M));
    G.tiles_n = int32_t(ceil_div(G.N, tc::BN));
    G.tiles_per_mat = G.syrk ? syrk_tiles(G.M) : G.tiles_m * G.tiles_n;
    G.tile_begin = tiles;
    const int64_t t64 = int64_t(tiles) + int64_t(G.tiles_per_mat) * G.count;
    if (t64 > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
    tiles = int(t64);
  }
  p.total_tiles = tiles;
  if (last && stage == NS_APPLY && std::isfinite(update_alpha)) {
    p.stage = TC_UPDATE;
    p.a = update_alpha;
    for (int g = 0; g < p.ngroups; ++g) p.g[g].alpha = update_alpha;
  }
  return tc_gemm_launch(p, stream);
}

mao_status run_simt_stage(const Buffers& buf, const std::vector<const NsGroupPlan*>& round,
                          int stage, int cur, bool first, bool last, const float* co,
                          const float* scale, const OutEntry* table, cudaStream_t stream) {
  SimtParams p;
  memset(&p, 0, sizeof(p));
  p.ngroups = int32_t(round.size());
  p.stage = stage;
  p.a = co[0];
  p.b = co[1];
  p.c = co[2];
  p.scale = first ? scale : nullptr;
  p.out_table = table;
  int64_t blocks = 0;
  for (size_t gi = 0; gi < round.size(); ++gi) {
    const NsGroupPlan& g = *round[gi];
    SimtGroup& G = p.g[gi];
    G.count = g.count;
    G.slot0 = g.slot0;
    G.orig_cols = int32_t(g.C);
    const float* X = reinterpret_cast<const float*>(buf.x(g, cur));
    const float* Ab = reinterpret_cast<const float*>(buf.a(g));
    const float* Bb = reinterpret_cast<const float*>(buf.b(g));
    const int64_t xs = g.R * g.ldx, as = g.m * g.lda;
    if (stage == NS_GRAM) {
      G.a = G.b = X;
      G.a_ms = G.b_ms = xs;
      if (!g.tall) { G.a_si = G.b_sj = g.ldx; G.a_sk = G.b_sk = 1; }
      else { G.a_si = G.b_sj = 1; G.a_sk = G.b_sk = g.ldx; }
      G.M = G.N = int32_t(g.m);
      G.K = int32_t(g.n);
      G.out = reinterpret_cast<float*>(buf.a(g));
      G.out_ld = g.lda;
      G.out_ms = as;
      G.res = Ab;
      G.syrk = 1;
    } else if (stage == NS_POLY) {
      G.a = G.b = Ab;
      G.a_ms = G.b_ms = as;
      G.a_si = G.b_sj = g.lda;
      G.a_sk = G.b_sk = 1;
      G.M = G.N = G.K = int32_t(g.m);
      G.out = reinterpret_cast<float*>(buf.b(g));
      G.out_ld = g.lda;
      G.out_ms = as;
      G.res = Ab;
      G.res_ld = g.lda;
      G.res_ms = as;
      G.syrk = 1;
    } else {
      if (!g.tall) {
        G.a = Bb; G.a_ms = as; G.a_si = g.lda; G.a_sk = 1;
        G.b = X;  G.b_ms = xs; G.b_sj = 1;     G.b_sk = g.ldx;
      } else {
        G.a = X;  G.a_ms = xs; G.a_si = g.ldx; G.a_sk = 1;
        G.b = Bb; G.b_ms = as; G.b_sj = g.lda; G.b_sk = 1;
      }
      G.M = int32_t(g.R);
      G.N = int32_t(g.C);
      G.K = int32_t(g.m);
      G.out = last ? nullptr : reinterpret_cast<float*>(buf.x(g, 1 - cur));
      G.out_ld = g.ldx;
      G.out_ms = xs;
      G.res = X;
      G.res_ld = g.ldx;
      G.res_ms = xs;
      G.syrk = 0;
      G.final_out = last ? 1 : 0;
    }
    G.tiles_m = int32_t(ceil_div(G.M, kSimtTile));
    G.tiles_n = int32_t(ceil_div(G.N, kSimtTile));
    G.block_begin = blocks;
    blocks += int64_t(G.tiles_m) * G.tiles_n * G.count;
  }
  if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
  ns_simt_kernel<<<unsigned(blocks), 256, 0, stream>>>(p);
  count_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace

mao_status ns_run(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                  const float* coeffs, int32_t coeff_stride, float eps, int32_t compute,
                  uint32_t* const* sign_bits, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream, const NsFuse* fuse) {
  NsPlan plan;
  make_ns_plan(in, batch, compute, plan);
  if (workspace_bytes < plan.total) return MAO_ERR_WORKSPACE;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  OutEntry* table = reinterpret_cast<OutEntry*>(ws + plan.off_out_table);
  float* scale = reinterpret_cast<float*>(ws + plan.off_scale);
  float* partials = reinterpret_cast<float*>(ws + plan.off_partials);
  int64_t* prange = reinterpret_cast<int64_t*>(ws + plan.off_prange);
  const bool tcpath = compute == MAO_BF16;
  const int32_t ws_dt = tcpath ? MAO_BF16 : MAO_F32;
  if (fuse && (!tcpath || (fuse->update && sign_bits))) return MAO_ERR_UNSUPPORTED;
  const bool upd = fuse && fuse->update;  // the last product updates out in place
  // small fp32 matrices: the whole call in one launch, one cluster per matrix. The choice
  // is made per matrix, so a matrix's result does not depend on the rest of the batch.
  if (!fuse && compute == MAO_F32) {
    std::vector<mao_mat> in_s, out_s, in_r, out_r;
    std::vector<uint32_t*> bits_s, bits_r;
    for (int b = 0; b < batch; ++b) {
      const bool small = ns_small_eligible(&in[b], &out[b], 1, steps, compute);
      (small ? in_s : in_r).push_back(in[b]);
      (small ? out_s : out_r).push_back(out[b]);
      (small ? bits_s : bits_r).push_back(sign_bits ? sign_bits[b] : nullptr);
    }
    if (!in_s.empty()) {
      const mao_status st =
          ns_small_run(in_s.data(), out_s.data(), int32_t(in_s.size()), steps, coeffs,
                       coeff_stride, eps, sign_bits ? bits_s.data() : nullptr, stream);
      if (st != MAO_OK || in_r.empty()) return st;
      return ns_run(in_r.data(), out_r.data(), int32_t(in_r.size()), steps, coeffs, coeff_stride,
                    eps, compute, sign_bits ? bits_r.data() : nullptr, workspace,
                    workspace_bytes, stream, nullptr);
    }
  }

  // ---- output entries; sign buffers filled by atomics start from zero
  std::vector<OutEntry> entries(batch);
  for (int b = 0; b < batch; ++b) {
    OutEntry& e = entries[b];
    e.src = upd && fuse->W_in ? fuse->W_in[b].data : nullptr;
    e.src_ld = upd && fuse->W_in ? fuse->W_in[b].ld : 0;
    e.out = out[b].data;
    e.bits = sign_bits ? sign_bits[b] : nullptr;
    e.ld = out[b].ld;
    e.dtype = out[b].dtype;
    e.flags = 0;
    if (e.out && (reinterpret_cast<uintptr_t>(e.out) % 16 == 0) &&
        ((out[b].ld * elem_size(out[b].dtype)) % 16 == 0) &&
        (!e.src || (reinterpret_cast<uintptr_t>(e.src) % 16 == 0 &&
                    (e.src_ld * elem_size(out[b].dtype)) % 16 == 0)))
      e.flags |= OUT_VEC;
    if (tcpath && in[b].cols % 32 == 0) e.flags |= OUT_WORDS;
    if (e.bits && !(e.flags & OUT_WORDS)) {
      const int64_t words = ceil_div(in[b].rows * in[b].cols, 32);
      if (cudaMemsetAsync(e.bits, 0, size_t(words) * 4, stream) != cudaSuccess) return MAO_ERR_CUDA;
    }
  }

  // ---- stage-in (copy to the workspace, partial sums of squares), in launches of kStageMax
  {
    int s = 0;
    while (s < batch) {
      StageParams p;
      memset(&p, 0, sizeof(p));
      p.ws_dt = ws_dt;
      p.mu = fuse ? fuse->mu : 0.0f;
      p.table = table;
      p.prange = prange;
      p.partials = partials;
      int64_t blocks = 0;
      while (s < batch && p.n < kStageMax) {
        const int b = plan.input_of[s];
        const NsGroupPlan* gp = nullptr;
        for (const auto& g : plan.groups)
          if (s >= g.slot0 && s < g.slot0 + g.count) gp = &g;
        StageEntry& e = p.e[p.n++];
        e.src = in[b].data;
        e.src_ld = in[b].ld;
        e.src_dt = in[b].dtype;
        if (in[b].dtype == MAO_I8)
          e.vec_src = (reinterpret_cast<uintptr_t>(in[b].data) % 8 == 0 && in[b].cols % 8 == 0 &&
                       in[b].ld % 8 == 0) ? 1 : 0;
        else if (in[b].dtype == MAO_SIGN1)
          e.vec_src = 0;
        else
          e.vec_src = vec8_ok(in[b]) && (!fuse || vec8_ok(fuse->G[b])) ? 1 : 0;
        if (fuse) {
          e.g = fuse->G[b].data;
          e.g_ld = fuse->G[b].ld;
          e.g_dt = fuse->G[b].dtype;
        }
        e.dst = ws + gp->off_x[0] + size_t(s - gp->slot0) * size_t(gp->R * gp->ldx) * plan.es;
        e.dst_ld = gp->ldx;
        e.rows = in[b].rows;
        e.cols = in[b].cols;
        e.units_per_row = gp->ldx / 8;
        e.units = e.units_per_row * in[b].rows;
        e.block_begin = blocks;
        e.partial0 = plan.partial_begin[s];
        e.nblocks = ceil_div(e.units, kStageUnitsPerBlock);
        e.out = entries[b];
        e.slot = s;
        blocks += ceil_div(e.units, kStageUnitsPerBlock);
        ++s;
      }
      if (blocks > 0x7FFFFFFF) return MAO_ERR_UNSUPPORTED;
      stage_in_kernel<<<unsigned(blocks), kStageThreads, 0, stream>>>(p);
      count_launch();
      if (cudaGetLastError() != cudaSuccess) return MAO_ERR_CUDA;
    }
  }
  // ---- per-slot scale s = 1 / (||X||_F + eps)
  finalize_scale_kernel<<<unsigned(batch), 32, 0, stream>>>(partials, prange, scale, eps);
  count_launch();
  if (cudaGetLastError() != cudaSuccess) return MAO_ERR_CUDA;

  // ---- the iterations, for rounds of up to eight shape groups
  if (tcpath) profile_span_begin(stream);
  const Buffers buf{ws, &plan};
  const int max_groups = tcpath ? tc::MAX_GROUPS : kSimtMaxGroups;
  for (size_t g0 = 0; g0 < plan.groups.size(); g0 += max_groups) {
    std::vector<const NsGroupPlan*> round;
    for (size_t g = g0; g < plan.groups.size() && round.size() < size_t(max_groups); ++g)
      round.push_back(&plan.groups[g]);
    // the last product writes every U of the round as bf16 rows with 16-byte stores when
    // all of them allow it and none asks for signs
    int out_mode = tc::OUT_CALLER_BF16;
    for (const NsGroupPlan* g : round)
      for (int k = 0; k < g->count; ++k) {
        const OutEntry& e = entries[plan.input_of[g->slot0 + k]];
        if (!e.out || e.bits || e.dtype != MAO_BF16 || !(e.flags & OUT_VEC)) out_mode = tc::OUT_CALLER;
      }
    for (int it = 0; it < steps; ++it) {
      const float* co = coeffs + (coeff_stride ? 3 * it : 0);
      const int cur = it & 1;
      const bool first = it == 0, last = it == steps - 1;
      for (int stage = NS_GRAM; stage <= NS_APPLY; ++stage) {
        const mao_status st =
            tcpath ? run_tc_stage(buf, round, stage, cur, first, last, co, scale, table, out_mode,
                                  stream, upd ? -fuse->lr : NAN)
                   : run_simt_stage(buf, round, stage, cur, first, last, co, scale, table, stream);
        if (st != MAO_OK) return st;
      }
    }
  }
  if (tcpath) profile_span_end(stream);
  return MAO_OK;
}

}  // namespace mao
