// Grouped Newton–Schulz products on the 5th-generation tensor cores (sm_103a).
//
// One persistent kernel serves all three products of an iteration (the stage is a launch
// parameter):
//   NS_GRAM   A = alpha * X X^T            (symmetric: upper tiles + mirrored store)
//   NS_POLY   B = a I + b A + c A A        (symmetric; A A = A A^T by symmetry)
//   NS_APPLY  X' = beta * B X              (X . B in the tall orientation; B symmetric)
// a X + (b A + c A^2) X is evaluated as (a I + b A + c A^2) X: the identity term is added
// on the diagonal in the second product's epilogue, so the bf16 operand B rounds a + (...)
// rather than (...) alone, and the third product needs no residual read.
// over every matrix of up to eight shape groups. Each CTA owns one SM and walks a static
// stride of the flattened tile list.
//
// Roles per CTA (192 threads):
//   warp 0       TMA producer: 64x64 bf16 boxes with 128-byte swizzle into a 4-stage ring
//   warp 1       allocates 512 TMEM columns; one thread issues tcgen05.mma (M=128, N<=256,
//                K=16, bf16 x bf16 -> fp32) and tcgen05.commit to release stages / tiles
//   warps 2..5   epilogue: tcgen05.ld of their 32-lane quadrant, fp32 arithmetic, stores
// The accumulator is double-buffered in TMEM so the epilogue of one tile overlaps the
// main loop of the next. Every barrier wait is bounded (globaltimer); a wait that gives up
// sets the device error word, drains the copies and products in flight, frees TMEM and
// returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ns_plan.h"

namespace mao {

__device__ unsigned int g_tc_error;  // bit 0: a barrier wait timed out

#ifdef MAO_TC_TRACE
// Debug builds only: cycles each role spends waiting, summed over CTAs.
// [0] producer waiting for a free stage, [1] MMA waiting for data, [2] MMA waiting for a
// free accumulator, [3] epilogue waiting for an accumulator, [4] epilogue busy cycles,
// [5] MMA k-blocks, [6] tiles, [7] total CTA cycles
__device__ unsigned long long g_tc_trace[16];
#define TRACE_T0() const long long _t0 = clock64()
#define TRACE_ADD(i, t0) atomicAdd(&g_tc_trace[i], (unsigned long long)(clock64() - (t0)))
#else
#define TRACE_T0()
#define TRACE_ADD(i, t0)
#endif

namespace {

using namespace tc;

// ----------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test with cluster-scope acquire (for barriers another CTA of the cluster arrives on).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete. Gives up after `limit_ns` or when another
// role raised the CTA's abort flag; a timeout sets the abort flag and the error word.
template <bool CLUSTER = false>
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint64_t limit_ns) {
  auto test = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (test()) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(&g_tc_error, 1u);
      return false;
    }
  }
}

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, fixed version field 0b001 at bit 46.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(lbo >> 4) << 16) |
         (uint64_t(sbo >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, M = 128.
__device__ __forceinline__ uint32_t instr_desc(int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(n >> 3) << 17) | (uint32_t(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape), waited on.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Issues a 32-column TMEM load without waiting; tmem_wait32 completes it. The wait takes
// the destination registers as operands so no use can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ------------------------------------------------------------------ tile walk

struct Tile {
  int g, z, row0, col0, m_valid, n_valid, nkb;
};

template <int TM>
__device__ __forceinline__ void decode_tile_t(const TcParams& p, int tile, Tile& t) {
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= tile) ++g;
  const TcGroup& G = p.g[g];
  const int local = tile - G.tile_begin;
  t.g = g;
  t.z = local / G.tiles_per_mat;
  int r = local - t.z * G.tiles_per_mat;
  if (G.syrk) {
    // row block ib covers columns [TM ib, N) in 256-wide tiles (upper triangle)
    int ib = 0;
    while (true) {
      const int cnt = (G.N - TM * ib + BN - 1) / BN;
      if (r < cnt) break;
      r -= cnt;
      ++ib;
    }
    t.row0 = TM * ib;
    t.col0 = TM * ib + BN * r;
  } else {
    const int tm = r / G.tiles_n;
    t.row0 = tm * TM;
    t.col0 = (r - tm * G.tiles_n) * BN;
  }
  t.m_valid = min(TM, G.M - t.row0);
  t.n_valid = min(BN, G.N - t.col0);
  t.nkb = (G.K + BK - 1) / BK;
}

__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, Tile& t) {
  decode_tile_t<BM>(p, tile, t);
}

// ------------------------------------------------------------------ epilogue

__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src, bool full, int nvalid,
                                            float (&v)[32]) {
  if (full) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + 8 * q);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[8 * q + 2 * i] = f.x;
        v[8 * q + 2 * i + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < nvalid ? __bfloat162float(src[i]) : 0.0f;
  }
}

// 32 bf16 values kept packed (16 registers) until used; zeros where out of range.
__device__ __forceinline__ void load32_packed(const __nv_bfloat16* src, bool full, int nvalid,
                                              uint4 (&q)[4]) {
  if (full) {
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = *reinterpret_cast<const uint4*>(src + 8 * k);
  } else {
    __nv_bfloat16 tmp[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) tmp[c] = c < nvalid ? src[c] : __float2bfloat16_rn(0.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = reinterpret_cast<const uint4*>(tmp)[k];
  }
}

__device__ __forceinline__ void unpack32(const uint4 (&q)[4], float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q[k]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * k + 2 * i] = f.x;
      v[8 * k + 2 * i + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 raw;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
    *reinterpret_cast<uint4*>(dst + 8 * q) = raw;
  }
}

// Symmetric store of one warp's 32x32 chunk (rows i0.., columns j0..) of the product:
// element (i, j) is written at (i, j) when j >= i and at (j, i) when j > i, so each stored
// pair comes from one accumulator value and the result is exactly symmetric.
__device__ __forceinline__ void store_sym_chunk(__nv_bfloat16* out, int64_t ld, int M, int i0,
                                                int j0, int lane, const float (&w)[32],
                                                __nv_bfloat16 (*tp)[TPAD]) {
  const int i = i0 + lane;
  const bool above = j0 >= i0 + 32;  // whole chunk strictly above the diagonal
  // direct rows
  if (i < M) {
    __nv_bfloat16* dst = out + int64_t(i) * ld + j0;
    if (above && j0 + 32 <= M) {
      store32_bf16(dst, w);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int j = j0 + c;
        if (j < M && j >= i) dst[c] = __float2bfloat16_rn(w[c]);
      }
    }
  }
  // mirrored rows through a shared-memory transpose
#pragma unroll
  for (int c = 0; c < 32; ++c) tp[lane][c] = __float2bfloat16_rn(w[c]);
  __syncwarp();
  const int j = j0 + lane;  // this thread writes row j of the mirror, columns i0..i0+31
  if (j < M) {
    __nv_bfloat16* dst = out + int64_t(j) * ld + i0;
    if (above && i0 + 32 <= M) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 raw;
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&raw);
#pragma unroll
        for (int r = 0; r < 8; ++r) h[r] = tp[8 * q + r][lane];
        *reinterpret_cast<uint4*>(dst + 8 * q) = raw;
      }
    } else {
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const int ii = i0 + r;
        if (ii < M && j > ii) dst[r] = tp[r][lane];
      }
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void store_final(const OutEntry& e, int i, int j0, int nvalid,
                                            int orig_cols, const float (&w)[32]) {
  if (e.out) {
    const int64_t base = int64_t(i) * e.ld + j0;
    if ((e.flags & OUT_VEC) && nvalid == 32) {
      if (e.dtype == MAO_BF16) {
        store32_bf16(reinterpret_cast<__nv_bfloat16*>(e.out) + base, w);
      } else {
        float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + base);
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = make_float4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) store_elem(e.out, base + c, e.dtype, w[c]);
    }
  }
  if (e.bits) {
    if (e.flags & OUT_WORDS) {  // C % 32 == 0: the 32 columns are one word
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 32; ++c) word |= (w[c] < 0.0f ? 0u : 1u) << c;
      e.bits[(int64_t(i) * orig_cols + j0) >> 5] = word;
    } else {  // words straddle rows: set bits into a zeroed buffer
#pragma unroll 1
      for (int c = 0; c < nvalid; ++c) {
        if (!(w[c] < 0.0f)) {
          const int64_t k = int64_t(i) * orig_cols + j0 + c;
          atomicOr(e.bits + (k >> 5), 1u << (k & 31));
        }
      }
    }
  }
}

// ------------------------------------------------------------------ the kernel

__global__ void __launch_bounds__(THREADS, 1) ns_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __nv_bfloat16(*tpose)[32][TPAD] =
      reinterpret_cast<__nv_bfloat16(*)[32][TPAD]>(smem + STAGES * STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + 4 * 32 * TPAD * 2);
  uint64_t* full_bar = bars;                 // [STAGES]  TMA -> MMA
  uint64_t* empty_bar = bars + STAGES;       // [STAGES]  MMA -> TMA
  uint64_t* tfull_bar = bars + 2 * STAGES;   // [2]       MMA -> epilogue
  uint64_t* tempty_bar = tfull_bar + 2;      // [2]       epilogue -> MMA
  uint64_t* drain_bar = tempty_bar + 2;      // [1]       MMA drain after an abort
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
#ifdef MAO_TC_TRACE
  __shared__ volatile long long arm_time[STAGES];
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 4);
    }
    mbar_init(smem_u32(drain_bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint64_t limit = p.timeout_ns;
#ifdef MAO_TC_TRACE
  const long long t_cta = clock64();
#endif

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for a free stage and arms its barrier; then lane q issues box q of the
    // stage (A boxes first, then B boxes), so the boxes of one stage are issued in parallel.
#ifndef MAO_TC_NO_DESC_PREFETCH
    if (lane == 0) {
      for (int g = 0; g < p.ngroups; ++g) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.g[g].tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.g[g].tmB)) : "memory");
      }
    }
#endif
    int stage = 0;
    uint32_t phase = 0;
    int armed_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) armed_parity[s] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
      Tile t;
      decode_tile(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int abox = G.a_box_rows, bbox = G.b_box_rows;
      const int nbox_a = BM / abox;
      const int nbox_b = (t.n_valid + bbox - 1) / bbox;
      const uint32_t bytes = uint32_t(nbox_a * abox + nbox_b * bbox) * 128u;
      // this lane's box: operand, tensor map, destination offset and tile coordinate
      const bool is_a = lane < nbox_a;
      const bool active = lane < nbox_a + nbox_b;
      const int q = is_a ? lane : lane - nbox_a;
      const CUtensorMap* map = is_a ? &G.tmA : &G.tmB;
      const int mn = is_a ? G.a_mn : G.b_mn;
      const int box = is_a ? abox : bbox;
      const uint32_t off = (is_a ? 0u : uint32_t(A_STAGE_BYTES)) + uint32_t(q * box) * 128u;
      const int rc = (is_a ? t.row0 : t.col0) + box * q;
      for (int kb = 0; kb < t.nkb; ++kb) {
        int okw = 1;
        if (lane == 0) {
#ifdef MAO_TC_TRACE
          const long long tw = clock64();
#endif
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, limit)) {
            okw = 0;
          } else {
            TRACE_ADD(0, tw);
            mbar_expect_tx(smem_u32(&full_bar[stage]), bytes);
            armed_parity[stage] = int(phase);
#ifdef MAO_TC_TRACE
            arm_time[stage] = clock64();
#endif
          }
        }
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
#ifdef MAO_TC_TRACE
        const long long t_tma = clock64();
#endif
        if (active) {
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const uint32_t dst = smem_u32(ring + stage * STAGE_BYTES) + off;
          const int k0 = kb * BK;
          if (mn) tma_load_3d(dst, map, fb, rc, k0, t.z);
          else tma_load_3d(dst, map, fb, k0, rc, t.z);
        }
#ifdef MAO_TC_TRACE
        __syncwarp();
        if (lane == 0) {
          atomicAdd(&g_tc_trace[10], (unsigned long long)(clock64() - t_tma));
          atomicAdd(&g_tc_trace[11], (unsigned long long)(nbox_a + nbox_b));
        }
#endif
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {  // let every copy in flight land before the CTA exits
      for (int s = 0; s < STAGES; ++s)
        if (armed_parity[s] >= 0) mbar_drain(smem_u32(&full_bar[s]), uint32_t(armed_parity[s]), 1000000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      bool issued = false;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++local) {
        Tile t;
        decode_tile(p, tile, t);
        const TcGroup& G = p.g[t.g];
        const int acc = local & 1;
        const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
#ifdef MAO_TC_TRACE
        const long long tw0 = clock64();
#endif
        if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        TRACE_ADD(2, tw0);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        const int n_mma = (t.n_valid + 15) & ~15;
        const uint32_t idesc = instr_desc(n_mma, G.a_mn, G.b_mn);
        for (int kb = 0; kb < t.nkb; ++kb) {
#ifdef MAO_TC_TRACE
          const long long tw1 = clock64();
#endif
          if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, limit)) {
            ok = false;
            break;
          }
          TRACE_ADD(1, tw1);
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[5], 1ull);
          const long long t_issue = clock64();
          atomicAdd(&g_tc_trace[9], (unsigned long long)(t_issue - arm_time[stage]));
#endif
#ifndef MAO_TC_NO_FULL_FENCE
          tc_fence_after();
#endif
          const uint32_t a_base = smem_u32(ring + stage * STAGE_BYTES);
          const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // K-major: 16 k-elements are 32 bytes along the swizzled row.
            // MN-major: 16 k-rows are two 1024-byte swizzle atoms.
            const uint64_t ad = G.a_mn ? smem_desc(a_base + kk * 2048, BOX_BYTES, 1024)
                                       : smem_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = G.b_mn ? smem_desc(b_base + kk * 2048, BOX_BYTES, 1024)
                                       : smem_desc(b_base + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            issued = true;
          }
          umma_commit(smem_u32(&empty_bar[stage]));
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[8], (unsigned long long)(clock64() - t_issue));
#endif
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull_bar[acc]));
      }
      if (!ok && issued) {  // wait for every product in flight before TMEM is freed
        umma_commit(smem_u32(drain_bar));
        mbar_drain(smem_u32(drain_bar), 0u, 1000000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    __nv_bfloat16(*tp)[TPAD] = tpose[warp - 2];
    int local = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++local) {
      Tile t;
      decode_tile(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int acc = local & 1;
      const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
#ifdef MAO_TC_TRACE
      const long long tw2 = clock64();
#endif
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, limit)) break;
      tc_fence_after();
#ifdef MAO_TC_TRACE
      if (lane == 0) TRACE_ADD(3, tw2);
      const long long tb = clock64();
#endif
      const int slot = G.slot0 + t.z;
      const float s = p.scale ? p.scale[slot] : 1.0f;
      const int rl = 32 * quad + lane;
      const int i = t.row0 + rl;
      const int i0 = t.row0 + 32 * quad;
      const bool row_ok = rl < t.m_valid;
      const int nchunks = (t.n_valid + 31) / 32;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(G.out) + int64_t(t.z) * G.out_mstride;
      const __nv_bfloat16* res =
          reinterpret_cast<const __nv_bfloat16*>(G.res) + int64_t(t.z) * G.res_mstride;
      OutEntry oe;
      if (G.final_out) oe = p.out_table[slot];
      const bool sym = p.stage != NS_APPLY;
      for (int cc = 0; cc < nchunks; ++cc) {
        const int j0 = t.col0 + 32 * cc;
        if (sym && j0 + 31 < i0) continue;  // strictly below the diagonal: mirrored elsewhere
        const int nvalid = min(32, G.N - j0);
        __syncwarp();
        float v[32];
        tmem_ld32(tmem_base + (uint32_t(32 * quad) << 16) + uint32_t(acc * BN + 32 * cc), v);
        if (sym) {
          float w[32];
          if (p.stage == NS_GRAM) {
            const float alpha = s * s;
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = alpha * v[c];
          } else {
            float r[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = 0.0f;
            if (row_ok) load32_bf16(res + int64_t(i) * G.res_ld + j0, nvalid == 32, nvalid, r);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              w[c] = __fmaf_rn(p.c, v[c], p.b * r[c]) + (j0 + c == i ? p.a : 0.0f);
          }
          store_sym_chunk(out, G.out_ld, G.M, i0, j0, lane, w, tp);
        } else if (row_ok) {
          float w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) w[c] = s * v[c];
          if (G.final_out) {
            store_final(oe, i, j0, nvalid, G.orig_cols, w);
          } else {
            __nv_bfloat16* dst = out + int64_t(i) * G.out_ld + j0;
            if (nvalid == 32) {
              store32_bf16(dst, w);
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < nvalid) dst[c] = __float2bfloat16_rn(w[c]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
#ifdef MAO_TC_TRACE
      if (lane == 0) {
        TRACE_ADD(4, tb);
        if (warp == 2) atomicAdd(&g_tc_trace[6], 1ull);
      }
#endif
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
#ifdef MAO_TC_TRACE
  if (threadIdx.x == 0) TRACE_ADD(7, t_cta);
#endif
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// The same three products with 256 x 256 tiles computed by a pair of CTAs on two SMs
// (thread-block cluster of 2, tcgen05 cta_group::2): CTA r holds rows [128 r, 128 r + 128)
// of the A operand tile and columns [128 r, 128 r + 128) of the B operand tile in its own
// shared memory; the even CTA issues M=256, N=256 products that read both halves, and each
// CTA's TMEM receives its 128 output rows. Per SM this moves 32 KB per 64-deep k-block
// instead of 48 KB, so a 6-stage ring fits. Barrier protocol:
//   full[s]   in the even CTA only: both CTAs' TMA loads complete their bytes on it; the
//             even CTA's producer arms it with the pair's total
//   empty[s]  in both CTAs: the even CTA's commit arrives on both (multicast)
//   tfull[a]  in both CTAs: commit multicast when an accumulator is complete
//   tempty[a] in the even CTA: the eight epilogue warps of the pair arrive on it

constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * 64 * 2;   // this CTA's A half: 128 rows x 64 k
constexpr int P_B_BYTES = 128 * 64 * 2;   // this CTA's B half: 128 columns x 64 k
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_TM = 256;                 // output rows per pair tile
#ifndef MAO_TC_EPI_WARPS
#define MAO_TC_EPI_WARPS 4
#endif
#ifndef MAO_TC_EPI_PIPE
#define MAO_TC_EPI_PIPE 0
#endif
constexpr int P_EPI_WARPS = MAO_TC_EPI_WARPS;  // 4 or 8 epilogue warps (one or two per TMEM quadrant)
constexpr int P_EPI_COLS = BN / (P_EPI_WARPS / 4);  // tile columns per epilogue warp
constexpr int P_EPI_CH = P_EPI_COLS / 32;           // 32-column chunks per epilogue warp
constexpr int P_THREADS = 64 + 32 * P_EPI_WARPS;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory, completing its bytes on a barrier that may live
// in the peer CTA (cta_group::2 form).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y,
                                                 int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the barrier at this shared-memory offset in every CTA of `mask` once all
// products issued so far by this thread are complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ uint32_t instr_desc_pair(int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(BN >> 3) << 17) | (uint32_t(P_TM >> 4) << 24);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    ns_tc_pair_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __nv_bfloat16(*tpose)[32][TPAD] =
      reinterpret_cast<__nv_bfloat16(*)[32][TPAD]>(smem + P_STAGES * P_STAGE_BYTES);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES + P_EPI_WARPS * 32 * TPAD * 2);
  uint64_t* full_bar = bars;                  // [P_STAGES]  (used in the even CTA)
  uint64_t* empty_bar = bars + P_STAGES;      // [P_STAGES]
  uint64_t* tfull_bar = bars + 2 * P_STAGES;  // [2]
  uint64_t* tempty_bar = tfull_bar + 2;       // [2]         (used in the even CTA)
  uint64_t* drain_bar = tempty_bar + 2;       // [1]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 2 * P_EPI_WARPS);
    }
    mbar_init(smem_u32(drain_bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint64_t limit = p.timeout_ns;
#ifdef MAO_TC_TRACE
  const long long t_cta = clock64();
#endif

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < p.total_tiles; tile += npairs) {
      Tile t;
      decode_tile_t<P_TM>(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int abox = G.a_box_rows, bbox = G.b_box_rows;
      const int nbox_a = 128 / abox, nbox_b = 128 / bbox;
      const bool is_a = lane < nbox_a;
      const bool active = lane < nbox_a + nbox_b;
      const int q = is_a ? lane : lane - nbox_a;
      const CUtensorMap* map = is_a ? &G.tmA : &G.tmB;
      const int mn = is_a ? G.a_mn : G.b_mn;
      const int box = is_a ? abox : bbox;
      const uint32_t off = (is_a ? 0u : uint32_t(P_A_BYTES)) + uint32_t(q * box) * 128u;
      const int rc = (is_a ? t.row0 : t.col0) + 128 * int(cta) + box * q;
      for (int kb = 0; kb < t.nkb; ++kb) {
        int okw = 1;
        if (lane == 0) {
#ifdef MAO_TC_TRACE
          const long long tw = clock64();
#endif
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, limit)) okw = 0;
          else if (leader) mbar_expect_tx(smem_u32(&full_bar[stage]), 2u * P_STAGE_BYTES);
#ifdef MAO_TC_TRACE
          if (leader) TRACE_ADD(0, tw);
#endif
        }
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        if (active) {
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
          const uint32_t dst = smem_u32(ring + stage * P_STAGE_BYTES) + off;
          const int k0 = kb * BK;
          if (mn) tma_load_3d_pair(dst, map, fb, rc, k0, t.z);
          else tma_load_3d_pair(dst, map, fb, k0, rc, t.z);
        }
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      bool issued = false;
      for (int tile = pair; ok && tile < p.total_tiles; tile += npairs, ++local) {
        Tile t;
        decode_tile_t<P_TM>(p, tile, t);
        const TcGroup& G = p.g[t.g];
        const int acc = local & 1;
        const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
#ifdef MAO_TC_TRACE
        const long long tw0 = clock64();
#endif
        if (!mbar_wait<true>(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        TRACE_ADD(2, tw0);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        const uint32_t idesc = instr_desc_pair(G.a_mn, G.b_mn);
        for (int kb = 0; kb < t.nkb; ++kb) {
#ifdef MAO_TC_TRACE
          const long long tw1 = clock64();
#endif
          if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, limit)) {
            ok = false;
            break;
          }
          TRACE_ADD(1, tw1);
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[5], 1ull);
          const long long t_issue = clock64();
#endif
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + stage * P_STAGE_BYTES);
          const uint32_t b_base = a_base + P_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = G.a_mn ? smem_desc(a_base + kk * 2048, BOX_BYTES, 1024)
                                       : smem_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = G.b_mn ? smem_desc(b_base + kk * 2048, BOX_BYTES, 1024)
                                       : smem_desc(b_base + kk * 32, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            issued = true;
          }
          umma_commit_pair(smem_u32(&empty_bar[stage]), 3);
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[8], (unsigned long long)(clock64() - t_issue));
#endif
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull_bar[acc]), 3);
      }
      if (!ok && issued) {
        umma_commit_pair(smem_u32(drain_bar), 1);
        mbar_drain(smem_u32(drain_bar), 0u, 1000000000ull);
      }
    }
    __syncwarp();
  } else {
#if MAO_TC_EPI_PIPE
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Eight warps: warp w reads TMEM lanes 32*(w%4).. (its rows) and handles one half of
    // the tile's 256 columns, four chunks of 32. The TMEM load (and, for the polynomial
    // product, the residual load) of chunk k+1 is in flight while chunk k is processed.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;  // which column slice of the tile (0 with 4 warps)
    __nv_bfloat16(*tp)[TPAD] = tpose[warp - 2];
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty_bar[0]), 0),
                                       mapa_shared(smem_u32(&tempty_bar[1]), 0)};
    int local = 0;
    for (int tile = pair; tile < p.total_tiles; tile += npairs, ++local) {
      Tile t;
      decode_tile_t<P_TM>(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int acc = local & 1;
      const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
      const int slot = G.slot0 + t.z;
      // per-tile values fetched before waiting for the accumulator
      const float s = p.scale ? p.scale[slot] : 1.0f;
      OutEntry oe;
      if (G.final_out) oe = p.out_table[slot];
      const int crow0 = t.row0 + 128 * int(cta);
      const int i0 = crow0 + 32 * quad;
      const int i = i0 + lane;
      const bool row_ok = i < G.M;
      const int jbase = t.col0 + P_EPI_COLS * half;
      const int nch = jbase < G.N ? min(P_EPI_CH, (G.N - jbase + 31) / 32) : 0;
      const bool sym = p.stage != NS_APPLY;
      const bool poly = p.stage == NS_POLY;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(G.out) + int64_t(t.z) * G.out_mstride;
      const __nv_bfloat16* res =
          reinterpret_cast<const __nv_bfloat16*>(G.res) + int64_t(t.z) * G.res_mstride;
      const __nv_bfloat16* res_row = res + int64_t(i) * G.res_ld;
      uint4 qa[4], qb[4];
      if (poly && nch > 0 && row_ok)
        load32_packed(res_row + jbase, G.N - jbase >= 32, G.N - jbase, qa);
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, limit)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (uint32_t(32 * quad) << 16) + uint32_t(acc * BN + P_EPI_COLS * half);
      uint32_t ra[32], rb[32];
      if (nch > 0) tmem_ld32_issue(tbase, ra);
#pragma unroll
      for (int k = 0; k < P_EPI_CH; ++k) {
        if (k < nch) {
          uint32_t(&rc)[32] = (k & 1) ? rb : ra;
          uint32_t(&rn)[32] = (k & 1) ? ra : rb;
          uint4(&qc)[4] = (k & 1) ? qb : qa;
          uint4(&qn)[4] = (k & 1) ? qa : qb;
          tmem_wait32(rc);
          const int j0 = jbase + 32 * k;
          if (k + 1 < nch) {
            tmem_ld32_issue(tbase + uint32_t(32 * (k + 1)), rn);
            if (poly && row_ok)
              load32_packed(res_row + j0 + 32, G.N - j0 - 32 >= 32, G.N - j0 - 32, qn);
          }
          const int nvalid = min(32, G.N - j0);
          float w[32];
          if (sym) {
            if (j0 + 31 >= i0) {  // chunks strictly below the diagonal are mirrored elsewhere
              if (!poly) {
                const float alpha = s * s;
#pragma unroll
                for (int c = 0; c < 32; ++c) w[c] = alpha * __uint_as_float(rc[c]);
              } else {
                float r[32];
                if (row_ok) unpack32(qc, r);
                else
#pragma unroll
                  for (int c = 0; c < 32; ++c) r[c] = 0.0f;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                  w[c] = __fmaf_rn(p.c, __uint_as_float(rc[c]), p.b * r[c]) +
                         (j0 + c == i ? p.a : 0.0f);
              }
              store_sym_chunk(out, G.out_ld, G.M, i0, j0, lane, w, tp);
            }
          } else if (row_ok) {
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = s * __uint_as_float(rc[c]);
            if (G.final_out) {
              store_final(oe, i, j0, nvalid, G.orig_cols, w);
            } else {
              __nv_bfloat16* dst = out + int64_t(i) * G.out_ld + j0;
              if (nvalid == 32) {
                store32_bf16(dst, w);
              } else {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                  if (c < nvalid) dst[c] = __float2bfloat16_rn(w[c]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
    }
  }

#else
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Four warps: warp w reads TMEM lanes 32*(w%4).. (its 32 rows of this CTA's half of
    // the tile) and walks the tile's columns in chunks of 32.
    const int quad = warp & 3;
    __nv_bfloat16(*tp)[TPAD] = tpose[warp - 2];
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty_bar[0]), 0),
                                       mapa_shared(smem_u32(&tempty_bar[1]), 0)};
    int local = 0;
    for (int tile = pair; tile < p.total_tiles; tile += npairs, ++local) {
      Tile t;
      decode_tile_t<P_TM>(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int acc = local & 1;
      const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
#ifdef MAO_TC_TRACE
      const long long tw2 = clock64();
#endif
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, limit)) break;
      tc_fence_after();
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) TRACE_ADD(3, tw2);
      const long long tb = clock64();
#endif
      const int slot = G.slot0 + t.z;
      const float s = p.scale ? p.scale[slot] : 1.0f;
      const int crow0 = t.row0 + 128 * int(cta);  // this CTA's first output row
      const int rl = 32 * quad + lane;
      const int i = crow0 + rl;
      const int i0 = crow0 + 32 * quad;
      const bool row_ok = i < G.M;
      const int nchunks = (t.n_valid + 31) / 32;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(G.out) + int64_t(t.z) * G.out_mstride;
      const __nv_bfloat16* res =
          reinterpret_cast<const __nv_bfloat16*>(G.res) + int64_t(t.z) * G.res_mstride;
      OutEntry oe;
      if (G.final_out) oe = p.out_table[slot];
      const bool sym = p.stage != NS_APPLY;
      for (int cc = 0; cc < nchunks; ++cc) {
        const int j0 = t.col0 + 32 * cc;
        if (sym && j0 + 31 < i0) continue;  // strictly below the diagonal: mirrored elsewhere
        const int nvalid = min(32, G.N - j0);
        __syncwarp();
        float v[32];
        tmem_ld32(tmem_base + (uint32_t(32 * quad) << 16) + uint32_t(acc * BN + 32 * cc), v);
        if (sym) {
          float w[32];
          if (p.stage == NS_GRAM) {
            const float alpha = s * s;
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = alpha * v[c];
          } else {
            float r[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = 0.0f;
            if (row_ok) load32_bf16(res + int64_t(i) * G.res_ld + j0, nvalid == 32, nvalid, r);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              w[c] = __fmaf_rn(p.c, v[c], p.b * r[c]) + (j0 + c == i ? p.a : 0.0f);
          }
          store_sym_chunk(out, G.out_ld, G.M, i0, j0, lane, w, tp);
        } else if (row_ok) {
          float w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) w[c] = s * v[c];
          if (G.final_out) {
            store_final(oe, i, j0, nvalid, G.orig_cols, w);
          } else {
            __nv_bfloat16* dst = out + int64_t(i) * G.out_ld + j0;
            if (nvalid == 32) {
              store32_bf16(dst, w);
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < nvalid) dst[c] = __float2bfloat16_rn(w[c]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) {
        TRACE_ADD(4, tb);
        if (warp == 2) atomicAdd(&g_tc_trace[6], 1ull);
      }
#endif
    }
  }

#endif
  tc_fence_before();
  __syncthreads();
#ifdef MAO_TC_TRACE
  if (threadIdx.x == 0 && leader) TRACE_ADD(7, t_cta);
#endif
  cluster_sync_all();  // no CTA leaves while its peer may still touch its shared memory
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

mao_status tc_encode_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                         int64_t ld, int64_t count, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return MAO_ERR_CUDA;
  const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), cuuint64_t(count)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2, cuuint64_t(rows) * cuuint64_t(ld) * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MAO_OK : MAO_ERR_UNSUPPORTED;
}

mao_status tc_gemm_launch(const TcParams& p, cudaStream_t stream) {
  if (p.total_tiles <= 0) return MAO_OK;
  static std::once_flag attr_once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(ns_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(SMEM_BYTES));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(ns_tc_pair_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(PAIR_SMEM_BYTES));
  });
  if (attr_err != cudaSuccess) return MAO_ERR_CUDA;
  profile_before_launch(stream);
  if (PAIR) {
    const int pairs = p.total_tiles < num_sms() / 2 ? p.total_tiles : num_sms() / 2;
    ns_tc_pair_kernel<<<2 * pairs, P_THREADS, PAIR_SMEM_BYTES, stream>>>(p);
  } else {
    const int grid = p.total_tiles < num_sms() ? p.total_tiles : num_sms();
    ns_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  }
  count_launch();
  profile_after_launch(stream);
  return cuda_status(cudaGetLastError());
}

#ifdef MAO_TC_TRACE
extern "C" int mao_debug_tc_trace(unsigned long long* out, int reset) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(out, g_tc_trace, sizeof(unsigned long long) * 16) != cudaSuccess) return -1;
  if (reset) {
    unsigned long long z[16] = {0};
    if (cudaMemcpyToSymbol(g_tc_trace, z, sizeof(z)) != cudaSuccess) return -1;
  }
  return 0;
}
#endif

mao_status tc_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_tc_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MAO_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MAO_ERR_CUDA;
  if (v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
      return MAO_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MAO_ERR_CUDA;
    return MAO_ERR_TIMEOUT;
  }
  return MAO_OK;
}

}  // namespace mao
