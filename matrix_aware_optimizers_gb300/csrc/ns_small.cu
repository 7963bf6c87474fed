// Newton–Schulz of small matrices on the fp32 accuracy path, the whole iteration in one
// launch.
//
// For a matrix whose working set (X twice, A, and this CTA's rows of B) fits in one SM's
// shared memory, the per-product launches of the general path cost more than the
// arithmetic. Here a cluster of sixteen CTAs owns one matrix for the whole call: every CTA
// holds all of X and A in shared memory and computes one sixteenth of the rows of each
// product ("分散ニュートン・シュルツ" of the Megatron Muon article: three products per
// iteration; the iteration of the Sign-Muon summary, §2 "Mecanismo Central" item 1):
//   A  = s^2 X X^T            rows of this CTA, sent to every other CTA
//   B' = a I + b A + c A A    rows of this CTA (local)
//   X' = s B' X               rows of this CTA into the other X buffer, sent likewise
// with s = 1/(||X||_F + eps) in the first iteration and 1 afterwards (the same placement
// of the normalisation as the general path). A CTA sends its rows with one bulk
// asynchronous copy per peer (shared memory to the peer's shared memory), whose bytes
// complete on the peer's barrier for that exchange; each CTA waits on its own barrier for
// the other fifteen CTAs' rows. No buffer is written while a peer may still read it: a CTA
// sends its A rows of the next iteration only after it holds every CTA's X rows of that
// iteration, which each CTA sends only after it has used the current A, and the X buffers
// alternate. Every CTA computes the Frobenius norm itself from its full copy in the same
// fixed order, so all sixteen hold the same s. At the end each CTA writes one sixteenth of
// U (in the matrix's own orientation) and of the packed signs, whole words, so the sign
// buffer needs no clearing. All arithmetic is fp32 FFMA with one accumulation chain per
// output, in k order.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ns_small.h"

namespace mao {
namespace {

constexpr int kCluster = 16;  // a non-portable cluster size (at most 8 is portable)
constexpr int kThreads = 256;

struct SmallEntry {
  const void* src;
  void* out;        // U (may be null)
  uint32_t* bits;   // packed signs (may be null)
  const void* g;    // with momentum: the gradient, and src (M) is updated in place
  int64_t src_ld, out_ld, g_ld;
  int32_t R, C, src_dt, out_dt, g_dt, pad;
};

struct SmallParams {
  SmallEntry e[kSmallMaxPerLaunch];
  float co[3 * 64];  // (a, b, c) of every iteration
  int32_t steps;
  float eps;
  int32_t momentum;  // M <- fma(mu, M, G), rounded to M's dtype, first; X = the new M
  float mu;
};

struct Layout {
  int m, n, nx, ma, rpc;
};

__host__ __device__ inline Layout layout_of(int R, int C) {
  Layout l;
  l.m = R < C ? R : C;
  l.n = R < C ? C : R;
  l.nx = ((l.n + 3) & ~3) + 4;  // X row stride (floats): 16-byte rows, conflict-free columns
  l.ma = ((l.m + 3) & ~3) + 4;  // A and B' row stride
  l.rpc = (l.m + kCluster - 1) / kCluster;
  return l;
}

__host__ __device__ inline size_t smem_floats(const Layout& l) {
  // X ping-pong, A, this CTA's rows of B', then 256 doubles for the norm's reduction
  return size_t(2) * l.m * l.nx + size_t(l.m) * l.ma + size_t(l.rpc) * l.ma + 2 * kThreads;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t remote(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ unsigned int g_small_error;  // bit 0: a row exchange did not complete in time

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Sends this CTA's rows [r0, r1) of buf (row stride ld floats, contiguous) to the same place
// in every other CTA of the cluster with bulk asynchronous copies, each completing its bytes
// on the receiver's barrier `bar` (same offset in every CTA). One thread issues them once
// every writer of the rows has fenced its writes for the async proxy and passed a CTA
// barrier; it waits until the copies have read the rows before returning, so the rows may
// be overwritten afterwards.
__device__ __forceinline__ void push_rows(const float* buf, int ld, int r0, int r1,
                                          uint64_t* bar, uint32_t self) {
  if (r1 <= r0) return;
  const uint32_t bytes = uint32_t(r1 - r0) * uint32_t(ld) * 4u;
  const uint32_t src = smem_addr(buf + size_t(r0) * ld);
  for (uint32_t q = 0; q < kCluster; ++q) {
    if (q == self) continue;
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(remote(src, q)), "r"(src), "r"(bytes), "r"(remote(smem_addr(bar), q))
        : "memory");
  }
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Arms this CTA's barrier for the bytes the other CTAs send in this phase (one arrival).
__device__ __forceinline__ void expect_rows(uint64_t* bar, int ld, int m, int own_rows) {
  const uint32_t bytes = uint32_t(m - own_rows) * uint32_t(ld) * 4u;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Waits (every thread) for the barrier's phase `parity`: the other CTAs' rows have landed.
// Bounded: after about 2 s the error word is set and the kernel goes on with what it has
// (wrong results, reported by mao_sync_status), so no wait can hang the GPU.
__device__ __forceinline__ void wait_rows(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  uint32_t ok = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  if (ok) return;
  const uint64_t t0 = globaltimer_ns();
  while (!ok) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (!ok && globaltimer_ns() - t0 > 2000000000ull) {
      atomicOr(&g_small_error, 1u);
      return;
    }
  }
}

// Four consecutive elements of a row as fp32 (k + 3 < n and `vec`: one 16-byte (f32) or
// 8-byte (bf16) load; otherwise element by element, zeros past n).
__device__ __forceinline__ float4 load4(const void* src, int64_t row_off, int k, int n, int dt,
                                        bool vec) {
  if (vec && k + 3 < n) {
    if (dt == MAO_BF16) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(
          reinterpret_cast<const __nv_bfloat16*>(src) + row_off + k));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      return make_float4(a.x, a.y, b.x, b.y);
    }
    return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + row_off + k));
  }
  float4 v;
  v.x = k < n ? load_elem(src, row_off + k, dt) : 0.0f;
  v.y = k + 1 < n ? load_elem(src, row_off + k + 1, dt) : 0.0f;
  v.z = k + 2 < n ? load_elem(src, row_off + k + 2, dt) : 0.0f;
  v.w = k + 3 < n ? load_elem(src, row_off + k + 3, dt) : 0.0f;
  return v;
}

// acc0 = sum_k P[i0][k] Q[j][k], acc1 = sum_k P[i1][k] Q[j][k] over kq quads (rows of
// stride ld floats, zero-padded to whole quads).
__device__ __forceinline__ void dot2(const float* P0, const float* P1, const float* Qj, int kq,
                                     float& acc0, float& acc1) {
  const float4* a = reinterpret_cast<const float4*>(P0);
  const float4* b = reinterpret_cast<const float4*>(P1);
  const float4* q = reinterpret_cast<const float4*>(Qj);
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 4
  for (int k = 0; k < kq; ++k) {
    const float4 x = q[k], u = a[k], v = b[k];
    s0 = __fmaf_rn(u.x, x.x, s0);
    s0 = __fmaf_rn(u.y, x.y, s0);
    s0 = __fmaf_rn(u.z, x.z, s0);
    s0 = __fmaf_rn(u.w, x.w, s0);
    s1 = __fmaf_rn(v.x, x.x, s1);
    s1 = __fmaf_rn(v.y, x.y, s1);
    s1 = __fmaf_rn(v.z, x.z, s1);
    s1 = __fmaf_rn(v.w, x.w, s1);
  }
  acc0 = s0;
  acc1 = s1;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    ns_small_kernel(const __grid_constant__ SmallParams p) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const SmallEntry& e = p.e[blockIdx.x / kCluster];
  const uint32_t crank = cluster_rank();
  const int tid = threadIdx.x;
  const bool tall = e.R > e.C;
  const Layout L = layout_of(e.R, e.C);
  const int m = L.m, n = L.n, nx = L.nx, ma = L.ma;
  const int r0 = min(m, int(crank) * L.rpc), r1 = min(m, r0 + L.rpc);  // this CTA's rows
  float* Xb[2] = {sm, sm + size_t(m) * nx};
  float* A = sm + size_t(2) * m * nx;
  float* Bm = A + size_t(m) * ma;
  double* red = reinterpret_cast<double*>(Bm + size_t(L.rpc) * ma);
  __shared__ uint64_t bar_a, bar_x;  // arrivals of the other CTAs' rows of A and of X
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar_a)) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar_x)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- the matrix into X[0] (X = M, or M^T for a tall M), zero-padded rows, and the sum of
  // squares in a fixed order (the same in every CTA of the cluster): per thread in fp32,
  // then the threads' sums in fp64
  float ss = 0.0f;
  // with momentum the matrix read is fma(mu, M, G) rounded to M's dtype (the stored new M)
  auto mom = [&](float mv, float gv) {
    const float v = __fmaf_rn(p.mu, mv, gv);
    return e.src_dt == MAO_BF16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
  };
  if (!tall) {
    const int es = e.src_dt == MAO_BF16 ? 2 : 4;
    const int gs = e.g_dt == MAO_BF16 ? 2 : 4;
    const bool vec = (reinterpret_cast<uintptr_t>(e.src) % (4 * es) == 0) && (e.src_ld % 4 == 0) &&
                     (!p.momentum || ((reinterpret_cast<uintptr_t>(e.g) % (4 * gs) == 0) && (e.g_ld % 4 == 0)));
    const int quads = nx / 4;  // the last quad of every row is padding
    constexpr int kU = 8;
    for (int t0 = tid; t0 < m * quads; t0 += kU * kThreads) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int t = t0 + u * kThreads;
        const int i = t / quads, q = t - i * quads;
        v[u] = t < m * quads ? load4(e.src, int64_t(i) * e.src_ld, 4 * q, n, e.src_dt, vec)
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      if (p.momentum) {  // every unit's G loads issued before any arithmetic
        float4 gv[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int t = t0 + u * kThreads;
          const int i = t / quads, q = t - i * quads;
          gv[u] = t < m * quads ? load4(e.g, int64_t(i) * e.g_ld, 4 * q, n, e.g_dt, vec)
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        // (zeros past n stay zero: fma(mu, 0, 0))
#pragma unroll
        for (int u = 0; u < kU; ++u)
          v[u] = make_float4(mom(v[u].x, gv[u].x), mom(v[u].y, gv[u].y), mom(v[u].z, gv[u].z),
                             mom(v[u].w, gv[u].w));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int t = t0 + u * kThreads;
        if (t < m * quads) {
          reinterpret_cast<float4*>(Xb[0])[t] = v[u];
          ss = __fmaf_rn(v[u].x, v[u].x, ss);
          ss = __fmaf_rn(v[u].y, v[u].y, ss);
          ss = __fmaf_rn(v[u].z, v[u].z, ss);
          ss = __fmaf_rn(v[u].w, v[u].w, ss);
        }
      }
    }
  } else {
    for (int idx = tid; idx < n * e.C; idx += kThreads) {  // source row-major: M[k][i]
      const int k = idx / e.C, i = idx - k * e.C;
      float v = load_elem(e.src, int64_t(k) * e.src_ld + i, e.src_dt);
      if (p.momentum) v = mom(v, load_elem(e.g, int64_t(k) * e.g_ld + i, e.g_dt));
      Xb[0][size_t(i) * nx + k] = v;
      ss = __fmaf_rn(v, v, ss);
    }
    for (int idx = tid; idx < m * (nx - n); idx += kThreads) {
      const int i = idx / (nx - n), k = n + idx - i * (nx - n);
      Xb[0][size_t(i) * nx + k] = 0.0f;
    }
  }
  for (int idx = tid; idx < m * (ma - m); idx += kThreads) {  // A's padding columns stay 0
    const int i = idx / (ma - m), k = m + idx - i * (ma - m);
    A[size_t(i) * ma + k] = 0.0f;
  }
  // fixed-order reduction: a shuffle tree within each warp, then the eight warp sums
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = double(ss);
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
  const float s = float(1.0 / (sqrt(tot) + double(p.eps)));
  // every CTA of the cluster is running, its barriers initialised, before any copy to it
  // (and with momentum, every CTA has read M before the new M is written over it)
  cluster_barrier();
  if (p.momentum) {  // the new M from X[0] (which iteration 0 only reads): this CTA's rows
    void* mo = const_cast<void*>(e.src);
    const int w = r1 - r0;
    for (int idx = tid; idx < w * n; idx += kThreads) {
      const int i = r0 + idx / n, k = idx % n;
      const int64_t at = tall ? int64_t(k) * e.src_ld + i : int64_t(i) * e.src_ld + k;
      store_elem(mo, at, e.src_dt, Xb[0][size_t(i) * nx + k]);
    }
  }

  const int xq = (n + 3) / 4, aq = (m + 3) / 4;
  const int pairs = (r1 - r0 + 1) / 2;
  for (int it = 0; it < p.steps; ++it) {
    const float ca = p.co[3 * it], cb = p.co[3 * it + 1], cc = p.co[3 * it + 2];
    const float* X = Xb[it & 1];
    float* Xn = Xb[(it + 1) & 1];
    const float s2 = it == 0 ? s * s : 1.0f;
    const float s1 = it == 0 ? s : 1.0f;
    const uint32_t parity = uint32_t(it) & 1u;
    // A = s^2 X X^T: rows i0, i0 + 1 of this CTA against row j, sent to every other CTA
    if (tid == 0) expect_rows(&bar_a, ma, m, r1 - r0);
    for (int t = tid; t < pairs * m; t += kThreads) {
      const int j = t % m, i0 = r0 + 2 * (t / m), i1 = min(i0 + 1, r1 - 1);
      float v0, v1;
      dot2(X + size_t(i0) * nx, X + size_t(i1) * nx, X + size_t(j) * nx, xq, v0, v1);
      A[size_t(i0) * ma + j] = s2 * v0;
      if (i0 + 1 < r1) A[size_t(i1) * ma + j] = s2 * v1;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) push_rows(A, ma, r0, r1, &bar_a, crank);
    wait_rows(&bar_a, parity);
    // B' = a I + b A + c A A (A A = A A^T): this CTA's rows, local
    for (int t = tid; t < pairs * m; t += kThreads) {
      const int j = t % m, i0 = r0 + 2 * (t / m), i1 = min(i0 + 1, r1 - 1);
      float v0, v1;
      dot2(A + size_t(i0) * ma, A + size_t(i1) * ma, A + size_t(j) * ma, aq, v0, v1);
      Bm[size_t(i0 - r0) * ma + j] =
          __fmaf_rn(cc, v0, cb * A[size_t(i0) * ma + j]) + (i0 == j ? ca : 0.0f);
      if (i0 + 1 < r1)
        Bm[size_t(i1 - r0) * ma + j] =
            __fmaf_rn(cc, v1, cb * A[size_t(i1) * ma + j]) + (i1 == j ? ca : 0.0f);
    }
    __syncthreads();
    // X' = s B' X: row i, columns 4q .. 4q + 3 (zeros past n), sent to every other CTA
    if (tid == 0) expect_rows(&bar_x, nx, m, r1 - r0);
    for (int t = tid; t < (r1 - r0) * xq; t += kThreads) {
      const int il = t / xq, q = t - il * xq;
      const float* brow = Bm + size_t(il) * ma;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
      for (int k = 0; k < m; ++k) {
        const float bv = brow[k];
        const float4 xv = reinterpret_cast<const float4*>(X + size_t(k) * nx)[q];
        acc.x = __fmaf_rn(bv, xv.x, acc.x);
        acc.y = __fmaf_rn(bv, xv.y, acc.y);
        acc.z = __fmaf_rn(bv, xv.z, acc.z);
        acc.w = __fmaf_rn(bv, xv.w, acc.w);
      }
      const int j = 4 * q;
      *reinterpret_cast<float4*>(Xn + size_t(r0 + il) * nx + j) =
          make_float4(s1 * acc.x, j + 1 < n ? s1 * acc.y : 0.0f, j + 2 < n ? s1 * acc.z : 0.0f,
                      j + 3 < n ? s1 * acc.w : 0.0f);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) push_rows(Xn, nx, r0, r1, &bar_x, crank);
    wait_rows(&bar_x, parity);
  }
  // every CTA has received all of its rows before any CTA leaves
  cluster_barrier();

  // ---- outputs from the final X (complete in every CTA): one sixteenth each
  const float* Xf = Xb[p.steps & 1];
  const int N = e.R * e.C;  // below 2^31: the working set fits one SM
  auto value = [&](int k) {  // entry k of U in its own row-major orientation
    const int r = k / e.C, c = k - r * e.C;
    return tall ? Xf[size_t(c) * nx + r] : Xf[size_t(r) * nx + c];
  };
  if (e.out) {
    const int per = (N + kCluster - 1) / kCluster;
    const int k0 = int(crank) * per, k1 = min(N, k0 + per);
    for (int k = k0 + tid; k < k1; k += kThreads) {
      const int r = k / e.C, c = k - r * e.C;
      store_elem(e.out, int64_t(r) * e.out_ld + c, e.out_dt, value(k));
    }
  }
  if (e.bits) {
    const int W = (N + 31) / 32;
    const int per = (W + kCluster - 1) / kCluster;
    const int w0 = int(crank) * per, w1 = min(W, w0 + per);
    for (int w = w0 + tid; w < w1; w += kThreads) {
      uint32_t word = 0;
      int r = (32 * w) / e.C, c = 32 * w - r * e.C;
      for (int b = 0; b < 32 && 32 * w + b < N; ++b) {
        const float v = tall ? Xf[size_t(c) * nx + r] : Xf[size_t(r) * nx + c];
        if (!(v < 0.0f)) word |= 1u << b;
        if (++c == e.C) {
          c = 0;
          ++r;
        }
      }
      e.bits[w] = word;
    }
  }
}

}  // namespace

mao_status small_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_small_error, sizeof(v), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return MAO_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MAO_ERR_CUDA;
  if (v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_small_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return MAO_ERR_CUDA;
    return MAO_ERR_TIMEOUT;
  }
  return MAO_OK;
}

size_t ns_small_smem_bytes(int64_t R, int64_t C) {
  if (R < 1 || C < 1 || R > 4096 || C > 4096) return ~size_t(0);
  return smem_floats(layout_of(int(R), int(C))) * sizeof(float);
}

// The kernel's attributes, set once per device: its shared memory and the non-portable
// cluster size; and whether a cluster of kCluster such CTAs can be placed at all (where it
// cannot, no matrix takes this path and the general one serves them).
bool small_kernel_ready() {
  static std::once_flag once[64];
  static bool ok[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::call_once(once[dev & 63], [&] {
    bool good =
        cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmallSmemMax)) == cudaSuccess;
    if (good) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(unsigned(kCluster));
      cfg.blockDim = dim3(unsigned(kThreads));
      cfg.dynamicSmemBytes = kSmallSmemMax;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      good = cudaOccupancyMaxActiveClusters(&clusters, ns_small_kernel, &cfg) == cudaSuccess &&
             clusters > 0;
    }
    cudaGetLastError();  // a refused query leaves no error behind for the caller
    ok[dev & 63] = good;
  });
  return ok[dev & 63];
}

bool ns_small_eligible(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                       int32_t compute) {
  if (compute != MAO_F32 || steps < 1 || steps > 64) return false;
  if (!small_kernel_ready()) return false;
  for (int b = 0; b < batch; ++b) {
    if (in[b].dtype != MAO_F32 && in[b].dtype != MAO_BF16) return false;
    if (ns_small_smem_bytes(in[b].rows, in[b].cols) > kSmallSmemMax) return false;
    if (out[b].data && out[b].dtype != MAO_F32 && out[b].dtype != MAO_BF16) return false;
  }
  return true;
}

mao_status ns_small_run(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                        const float* coeffs, int32_t coeff_stride, float eps,
                        uint32_t* const* sign_bits, cudaStream_t stream, const mao_mat* G,
                        float mu) {
  if (!small_kernel_ready()) return MAO_ERR_UNSUPPORTED;
  for (int b0 = 0; b0 < batch; b0 += kSmallMaxPerLaunch) {
    const int nb = std::min(batch - b0, kSmallMaxPerLaunch);
    SmallParams p;
    memset(&p, 0, sizeof(p));
    p.steps = steps;
    p.eps = eps;
    p.momentum = G ? 1 : 0;
    p.mu = mu;
    for (int it = 0; it < steps; ++it)
      for (int q = 0; q < 3; ++q) p.co[3 * it + q] = coeffs[(coeff_stride ? 3 * it : 0) + q];
    size_t smem = 0;
    for (int k = 0; k < nb; ++k) {
      const mao_mat& x = in[b0 + k];
      SmallEntry& e = p.e[k];
      e.src = x.data;
      e.src_ld = x.ld;
      e.src_dt = x.dtype;
      e.out = out[b0 + k].data;
      e.out_ld = out[b0 + k].ld;
      e.out_dt = out[b0 + k].dtype;
      e.bits = sign_bits ? sign_bits[b0 + k] : nullptr;
      e.R = int32_t(x.rows);
      e.C = int32_t(x.cols);
      if (G) {
        e.g = G[b0 + k].data;
        e.g_ld = G[b0 + k].ld;
        e.g_dt = G[b0 + k].dtype;
      }
      smem = std::max(smem, ns_small_smem_bytes(x.rows, x.cols));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(kCluster * nb));
    cfg.blockDim = dim3(unsigned(kThreads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    profile_before_launch(stream, MAO_PROF_NS_SMALL);
    const cudaError_t err = cudaLaunchKernelEx(&cfg, ns_small_kernel, p);
    count_launch();
    profile_after_launch(stream);
    if (err != cudaSuccess) return MAO_ERR_CUDA;
    const mao_status st = cuda_status(cudaGetLastError());
    if (st != MAO_OK) return st;
  }
  return MAO_OK;
}

}  // namespace mao
