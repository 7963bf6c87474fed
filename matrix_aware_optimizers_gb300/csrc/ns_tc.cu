// Grouped Newton–Schulz products on the 5th-generation tensor cores (sm_103a).
//
// One persistent kernel template serves all three products of an iteration (one
// instantiation per product, and one more for the last product of the last iteration, which
// writes the caller's outputs), over every matrix of up to eight shape groups:
//   NS_GRAM   A  = alpha * X X^T              (symmetric: upper and diagonal tiles only)
//   NS_POLY   B' = a I + b A + c A A          (symmetric; A A = A A^T by symmetry)
//   NS_APPLY  X' = beta * B' X                (X B' in the tall orientation; B' symmetric)
// and, for the Dion step, plain products into fp32 outputs (the final NS_APPLY
// instantiation with no scale) and an in-place rank-k update of the caller's matrices:
//   TC_UPDATE out <- out + a * (A B^T)
// which also serves as the last product of a fused Muon step (W <- W - lr U, U = B' X).
// A symmetric result is stored as its upper and diagonal 256 x 256 tiles. A product that
// reads it takes each 128-deep k-block below the diagonal from the transposed view of the
// stored upper block (an MN-major load of the same buffer), so no tile is ever mirrored.
// a X + (b A + c A^2) X is evaluated as (a I + b A + c A^2) X: the identity term is added
// on the diagonal in the second product's epilogue, so the bf16 operand rounds a + (...)
// rather than the cancelling (...) alone, and the third product reads no residual.
//
// Tiles of 256 x 256 outputs are computed by a pair of CTAs (thread-block cluster of two,
// tcgen05 cta_group::2). CTA r of the pair loads rows [128 r, 128 r + 128) of the A
// operand tile and columns [128 r, 128 r + 128) of the B operand tile into its own shared
// memory: per 128-deep k-block one 32 KB TMA box per operand half (64 columns x 128 rows x
// two 64-column chunks, 128-byte swizzle), a 3-stage ring of 64 KB; the even CTA issues
// M=256, N=256, K=16 products that read both halves; each CTA's TMEM receives its 128
// output rows (two 256-column fp32 accumulators, double-buffered).
//
// Roles per CTA (320 threads; 192 in the instantiations that write the caller's outputs):
//   warp 0       TMA producer: lane 0 waits for a free stage (and in the even CTA arms the
//                pair's full barrier); lanes 0 and 1 then issue the A and B boxes
//   warp 1       TMEM allocation (both CTAs); in the even CTA one thread issues tcgen05.mma
//                and multicasts tcgen05.commit to both CTAs' barriers
//   warps 2..9   epilogue: tcgen05.ld of their 32-lane quadrant (two warps per quadrant,
//                alternate 64-column blocks), fp32 arithmetic, then 32 x 64 blocks staged in
//                shared memory (128-byte swizzle) and written by bulk tensor stores; the
//                caller-output instantiations use warps 2..5, one per quadrant
// The in-place update (TC_UPDATE) reads and writes the caller's rows with 16-byte accesses
// from its eight epilogue warps. For a short product (K <= 256, a rank-k update) it runs as
// OUT_UPDATE_STREAM: a 2-stage operand ring, and per epilogue warp three 4 KB slots into
// which the warp copies (cp.async) the old values of its next blocks about a tile ahead.
// A long product (the last one of a fused Muon step) keeps the 3-stage ring and loads the
// old values into registers before its accumulator is ready.
// Barriers: full[s] (even CTA; both CTAs' loads complete on it), empty[s] (both CTAs),
// tfull[a] (both), tempty[a] (even CTA; every epilogue warp of the pair arrives on it).
// The kernel is launched as a programmatic dependent of the previous kernel in the stream:
// its set-up (barriers, TMEM) overlaps that kernel's tail.
// Every wait is bounded by %globaltimer (the limit is a launch parameter): a wait that
// gives up sets the device error word and the CTA's abort flag; the CTA then lets its
// in-flight loads (bounded waits on the armed stages), products (a drain commit) and stores
// land, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ns_plan.h"

namespace mao {

__device__ unsigned int g_tc_error;  // bit 0: a barrier wait timed out

#ifdef MAO_TC_TRACE
// Debug builds only: cycles the even CTA's roles spend waiting, summed over CTAs.
// [0] producer waiting for a free stage, [1] MMA waiting for data, [2] MMA waiting for a
// free accumulator, [3] epilogue waiting for an accumulator, [4] epilogue busy cycles,
// [5] MMA k-blocks, [6] tiles, [7] total CTA cycles, [8] MMA issue cycles
__device__ unsigned long long g_tc_trace[16];
#define TRACE_ADD(i, t0) atomicAdd(&g_tc_trace[i], (unsigned long long)(clock64() - (t0)))
#else
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

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Arrive on a barrier of the leader CTA. The signal it carries (this warp's TMEM reads are
// done) is ordered by tcgen05.fence::before_thread_sync, not by the arrive's memory
// semantics, so the arrive keeps the default CTA-scope release: a cluster-scope release
// would also wait for this thread's earlier global stores.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
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

// The same test with cluster-scope acquire (for barriers the peer CTA arrives on).
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

// Non-blocking test of the same phase (no suspension inside the instruction).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same non-blocking test with cluster-scope acquire.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete. Gives up after `limit_ns` or when another
// role raised the CTA's abort flag; a timeout sets the abort flag and the error word. A
// limit of 0 gives up at once unless a non-blocking test finds the phase complete (each
// try_wait may suspend the thread for a while, so polling alone could always succeed).
template <bool CLUSTER = false>
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint64_t limit_ns) {
  auto test = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (limit_ns == 0) {
    if (mbar_test_wait(bar, parity)) return true;
    *abort_flag = 1;
    atomicOr(&g_tc_error, 1u);
    return false;
  }
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

// mbar_wait with its common case inline: a phase that is already complete costs one
// non-blocking test and no call.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint64_t limit_ns) {
  const bool done = CLUSTER ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
  return done || mbar_wait<CLUSTER>(bar, parity, abort_flag, limit_ns);
}

// Bounded wait used only while draining after an abort (ignores the abort flag).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// TMA load into this CTA's shared memory, completing its bytes on a barrier that may live
// in the peer CTA (cta_group::2 form).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y,
                                                 int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar_cluster)
      : "memory");
}

// Bulk tensor store of a staged block (shared -> global) and its group bookkeeping.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
// Asks L2 to fetch the line holding `src` (through the load/store path: bulk prefetches
// would queue in the TMA unit behind, or ahead of, the operand loads).
__device__ __forceinline__ void prefetch_l2(const void* src) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(src) : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk store of this thread has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk store of this thread is complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's shared-memory writes before later async-proxy reads of them.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, M = 256, N = 256.
__device__ __forceinline__ uint32_t instr_desc(int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(BN >> 3) << 17) | (uint32_t(TILE_M >> 4) << 24);
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

// 64 consecutive fp32 columns of this thread's TMEM lane (32x32b shape, .x64): one load
// and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ tile walk

struct Tile {
  int g, z, row0, col0, n_valid, nkb;
};

// Tile `tile` of the flattened list: group, matrix, first output row and column.
// The k-th tile of CTA pair `pair`: tiles are dealt in rounds of npairs, round-robin, or
// with `snake` every other round in reverse pair order, so that with the deepest tiles listed
// first the pairs that drew the deeper tiles of a round draw the shallower ones of the next
// (products of mixed depths; the Newton–Schulz products, of even depth, keep round-robin,
// which measured faster for them).
__device__ __forceinline__ int pair_tile(int pair, int k, int npairs, int snake) {
  return k * npairs + ((snake & k & 1) ? npairs - 1 - pair : pair);
}

__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, Tile& t) {
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= tile) ++g;
  const TcGroup& G = p.g[g];
  const int local = tile - G.tile_begin;
  t.g = g;
  t.z = local / G.tiles_per_mat;
  int r = local - t.z * G.tiles_per_mat;
  if (G.syrk) {
    // row block ib covers columns [TILE_M ib, N) in 256-wide tiles (upper triangle)
    int ib = 0;
    while (true) {
      const int cnt = (G.N - TILE_M * ib + BN - 1) / BN;
      if (r < cnt) break;
      r -= cnt;
      ++ib;
    }
    t.row0 = TILE_M * ib;
    t.col0 = TILE_M * ib + BN * r;
  } else {
    const int tm = r / G.tiles_n;
    t.row0 = tm * TILE_M;
    t.col0 = (r - tm * G.tiles_n) * BN;
  }
  t.n_valid = min(BN, G.N - t.col0);
  t.nkb = (G.K + BK - 1) / BK;
}

// ------------------------------------------------------------------ epilogue
//
// Each epilogue warp owns 32 output rows i0..i0+31 (lane = row) and walks its share of the
// tile's columns in blocks of 64. A block's values pass through a per-warp staging buffer:
//   32 rows of 128 bytes; 16-byte chunk k of row r sits at chunk position k ^ (r & 7) (the
//   128-byte swizzle of the output's bulk-store map), so row-wise and column-wise accesses
//   of the warp hit distinct banks

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of 16-byte chunk k of row r in the row-major staging layout.
__device__ __forceinline__ int srow(int r, int k) { return r * 128 + ((k ^ (r & 7)) << 4); }

// Thread `lane` writes its row's 64 values (bf16) into the row-major staging buffer.
__device__ __forceinline__ void stage_rows(uint8_t* S, int lane, const float* w) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(S + srow(lane, k)) =
        make_uint4(pack_bf16x2(w[8 * k], w[8 * k + 1]), pack_bf16x2(w[8 * k + 2], w[8 * k + 3]),
                   pack_bf16x2(w[8 * k + 4], w[8 * k + 5]), pack_bf16x2(w[8 * k + 6], w[8 * k + 7]));
}

// Writes the staged 32 x 64 block to dst rows i0.., columns jb.. (row stride ld) with
// coalesced 16-byte stores; element (i, j) is written when i < M and j < ncols.
__device__ __forceinline__ void store_rows(const uint8_t* S, __nv_bfloat16* dst, int64_t ld,
                                           int i0, int jb, int M, int ncols, int lane) {
  const int sg = lane & 7;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = (lane >> 3) + 4 * q;
    const int gi = i0 + r;
    const int gj = jb + 8 * sg;
    if (gi >= M) continue;
    const uint4 val = *reinterpret_cast<const uint4*>(S + srow(r, sg));
    __nv_bfloat16* g = dst + int64_t(gi) * ld + gj;
    if (gj + 8 <= ncols) {
      *reinterpret_cast<uint4*>(g) = val;
    } else {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&val);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (gj + k < ncols) g[k] = e[k];
    }
  }
}

// The warp's 32 residual rows of a block (columns jb..jb+63) in row-contiguous 128-byte
// pieces: lane l holds 16-byte chunk l % 8 of rows l / 8 + 4 q (zeros past M). res_rows
// later turns them into one row per lane through the warp's staging buffer. Rows of the
// workspace are 128-byte aligned and zero-padded to a multiple of 64 columns, so the 64
// columns of a block are always addressable.
__device__ __forceinline__ void load_res_block(const __nv_bfloat16* src, int64_t ld, int i0,
                                               int jb, int M, int lane, uint4 (&r)[8]) {
  const __nv_bfloat16* base = src + jb + 8 * (lane & 7);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int gi = i0 + (lane >> 3) + 4 * q;
    r[q] = gi < M ? __ldg(reinterpret_cast<const uint4*>(base + int64_t(gi) * ld))
                  : make_uint4(0u, 0u, 0u, 0u);
  }
}

// r (load_res_block's layout) -> this lane's row, through the 4 KB staging buffer S.
__device__ __forceinline__ void res_rows(uint8_t* S, int lane, uint4 (&r)[8]) {
  const int sg = lane & 7;
#pragma unroll
  for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(S + srow((lane >> 3) + 4 * q, sg)) = r[q];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) r[k] = *reinterpret_cast<const uint4*>(S + srow(lane, k));
  __syncwarp();
}

// Element c (0..63) of a residual row held as eight 16-byte words.
__device__ __forceinline__ float res_elem(const uint4 (&r)[8], int c) {
  const uint4& u = r[c >> 3];
  const uint32_t w = (c & 7) < 2 ? u.x : (c & 7) < 4 ? u.y : (c & 7) < 6 ? u.z : u.w;
  return __uint_as_float((c & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// fp32 rows: this lane's row, columns jb..jb+63 (those below ncols), to dst. With vec (rows
// 16-byte aligned) two 32-column halves go through the staging buffer as 32 x 32 blocks of
// 128-byte rows; otherwise each lane writes its own row.
__device__ __forceinline__ void store_rows_f32(uint8_t* S, float* dst, int64_t ld, int i0, int jb, int M,
                                               int ncols, int lane, const float* w, bool vec) {
  if (vec) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4*>(S + srow(lane, k)) =
            make_float4(w[32 * h + 4 * k], w[32 * h + 4 * k + 1], w[32 * h + 4 * k + 2], w[32 * h + 4 * k + 3]);
      __syncwarp();
      const int sg = lane & 7;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int r = (lane >> 3) + 4 * q;
        const int gi = i0 + r;
        const int gj = jb + 32 * h + 4 * sg;
        if (gi >= M) continue;
        const float4 val = *reinterpret_cast<const float4*>(S + srow(r, sg));
        float* g = dst + int64_t(gi) * ld + gj;
        if (gj + 4 <= ncols) {
          *reinterpret_cast<float4*>(g) = val;
        } else {
          const float* f = reinterpret_cast<const float*>(&val);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (gj + k < ncols) g[k] = f[k];
        }
      }
      __syncwarp();
    }
  } else if (i0 + lane < M) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (jb + c < ncols) dst[int64_t(i0 + lane) * ld + jb + c] = w[c];
  }
}

// Final output of the last product for this lane's row, columns jb..jb+63: packed signs,
// an fp32 copy, and U through the slot's output entry, taken from the fp32 values w.
__device__ __forceinline__ void store_final(const OutEntry& e, uint8_t* S, int i0, int jb, int M,
                                            int N, int orig_cols, int lane, const float* w) {
  const int i = i0 + lane;
  if (e.bits && i < M) {
    if (e.flags & OUT_WORDS) {  // C % 32 == 0: each 32 columns are one word
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (jb + 32 * h < N) {
          uint32_t word = 0;
#pragma unroll
          for (int c = 0; c < 32; ++c) word |= (w[32 * h + c] < 0.0f ? 0u : 1u) << c;
          e.bits[(int64_t(i) * orig_cols + jb + 32 * h) >> 5] = word;
        }
      }
    } else {  // words straddle rows: set bits into a zeroed buffer
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        if (jb + c < N && !(w[c] < 0.0f)) {
          const int64_t k = int64_t(i) * orig_cols + jb + c;
          atomicOr(e.bits + (k >> 5), 1u << (k & 31));
        }
      }
    }
  }
  if (e.copy) store_rows_f32(S, e.copy, e.copy_ld, i0, jb, M, e.copy_cols, lane, w, (e.flags & OUT_COPY_VEC) != 0);
  if (!e.out) return;
  if ((e.flags & OUT_VEC) && e.dtype == MAO_BF16) {
    stage_rows(S, lane, w);
    __syncwarp();
    store_rows(S, reinterpret_cast<__nv_bfloat16*>(e.out), e.ld, i0, jb, M, N, lane);
    __syncwarp();
  } else if ((e.flags & OUT_VEC) && e.dtype == MAO_F32) {
    store_rows_f32(S, reinterpret_cast<float*>(e.out), e.ld, i0, jb, M, N, lane, w, true);
  } else if (i < M) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (jb + c < N) store_elem(e.out, int64_t(i) * e.ld + jb + c, e.dtype, w[c]);
  }
}

// TC_UPDATE on bf16 rows with 16-byte accesses: a warp's block (32 rows x 64 columns) moves
// between memory and registers in row-contiguous 128-byte pieces (8 lanes per row, four rows
// per instruction: lane l holds 16-byte chunk l % 8 of rows l / 8 + 4 q). The old values are
// loaded before the accumulator is ready; upd_apply turns them into the new values through
// the warp's staging buffer (one row per lane for the arithmetic), and upd_store writes them
// once the accumulator has been released. Both go around the L1 (L1::no_allocate): with the
// operand ring and staging in shared memory only a small L1 is left, and lines allocated for
// rows that are used once throttle the loads in flight.
__device__ __forceinline__ bool upd_block_vec(const OutEntry& e, int jb, int N) {
  return (e.flags & OUT_VEC) && e.dtype == MAO_BF16 && jb + 64 <= N;
}

// The old values of an update: e.src (row stride e.src_ld) or, when null, e.out itself.
__device__ __forceinline__ const void* upd_src(const OutEntry& e) { return e.src ? e.src : e.out; }
__device__ __forceinline__ int64_t upd_src_ld(const OutEntry& e) { return e.src ? e.src_ld : e.ld; }

__device__ __forceinline__ void upd_load(const OutEntry& e, int i0, int jb, int M, int lane,
                                         uint4 (&r)[8]) {
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(upd_src(e)) + jb + 8 * (lane & 7);
  const int64_t ld = upd_src_ld(e);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int gi = i0 + (lane >> 3) + 4 * q;
    if (gi < M) {
      uint4 v;
      asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "l"(base + int64_t(gi) * ld));
      r[q] = v;
    }
  }
}

__device__ __forceinline__ void upd_store(const OutEntry& e, int i0, int jb, int M, int lane,
                                          const uint4 (&r)[8]) {
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(e.out) + jb + 8 * (lane & 7);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int gi = i0 + (lane >> 3) + 4 * q;
    if (gi < M)
      asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(base + int64_t(gi) * e.ld),
                   "r"(r[q].x), "r"(r[q].y), "r"(r[q].z), "r"(r[q].w) : "memory");
  }
}

// r (old values, chunk layout of upd_load) -> new values fmaf(alpha, acc, old) rounded to
// bf16, same layout; w is this lane's row of the accumulator block.
__device__ __forceinline__ void upd_apply(uint8_t* S, int lane, const float* w, float alpha,
                                          uint4 (&r)[8]) {
  const int sg = lane & 7;
#pragma unroll
  for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(S + srow((lane >> 3) + 4 * q, sg)) = r[q];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint4 u = *reinterpret_cast<const uint4*>(S + srow(lane, k));
    uint32_t* h = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(h[q] << 16), hi = __uint_as_float(h[q] & 0xFFFF0000u);
      h[q] = pack_bf16x2(__fmaf_rn(alpha, w[8 * k + 2 * q], lo),
                         __fmaf_rn(alpha, w[8 * k + 2 * q + 1], hi));
    }
    *reinterpret_cast<uint4*>(S + srow(lane, k)) = u;
  }
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 8; ++q) r[q] = *reinterpret_cast<const uint4*>(S + srow((lane >> 3) + 4 * q, sg));
  __syncwarp();
}

// OUT_UPDATE_STREAM: the old values of a 32 x 64 block travel straight into a staging
// slot (16-byte cp.async per lane, same chunk layout as upd_load, L2 only), are turned
// into the new values in place (one row per lane), and leave with coalesced 16-byte stores.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void slot_fill(const OutEntry& e, uint8_t* S, int i0, int jb, int M,
                                          int lane) {
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(upd_src(e)) + jb + 8 * (lane & 7);
  const int64_t ld = upd_src_ld(e);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = (lane >> 3) + 4 * q;
    const int gi = i0 + r;
    if (gi < M) cp_async16(smem_u32(S + srow(r, lane & 7)), base + int64_t(gi) * ld);
  }
}

__device__ __forceinline__ void slot_apply(uint8_t* S, int lane, const float* w, float alpha) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint4 u = *reinterpret_cast<const uint4*>(S + srow(lane, k));
    uint32_t* h = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(h[q] << 16), hi = __uint_as_float(h[q] & 0xFFFF0000u);
      h[q] = pack_bf16x2(__fmaf_rn(alpha, w[8 * k + 2 * q], lo),
                         __fmaf_rn(alpha, w[8 * k + 2 * q + 1], hi));
    }
    *reinterpret_cast<uint4*>(S + srow(lane, k)) = u;
  }
}

__device__ __forceinline__ void slot_store(const OutEntry& e, const uint8_t* S, int i0, int jb,
                                           int M, int lane) {
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(e.out) + jb + 8 * (lane & 7);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = (lane >> 3) + 4 * q;
    const int gi = i0 + r;
    if (gi < M) {
      const uint4 v = *reinterpret_cast<const uint4*>(S + srow(r, lane & 7));
      asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(
                       base + int64_t(gi) * e.ld),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
  }
}

// Update of the caller's matrix for this lane's row, columns jb..jb+63:
// out = fmaf(alpha, acc, old) in fp32, rounded to out's dtype (old: upd_src).
__device__ __forceinline__ void update_final(const OutEntry& e, int i0, int jb, int M, int N,
                                             int lane, const float* w, float alpha) {
  const int i = i0 + lane;
  if (i >= M) return;
  const int64_t sld = upd_src_ld(e);
  if ((e.flags & OUT_VEC) && jb + 64 <= N) {
    if (e.dtype == MAO_BF16) {
      uint4* g = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(e.out) +
                                          int64_t(i) * e.ld + jb);
      const uint4* gs = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(upd_src(e)) + int64_t(i) * sld + jb);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 u = gs[k];
        uint32_t* h = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(h[q] << 16), hi = __uint_as_float(h[q] & 0xFFFF0000u);
          h[q] = pack_bf16x2(__fmaf_rn(alpha, w[8 * k + 2 * q], lo),
                             __fmaf_rn(alpha, w[8 * k + 2 * q + 1], hi));
        }
        g[k] = u;
      }
    } else {
      float4* g = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + int64_t(i) * e.ld + jb);
      const float4* gs =
          reinterpret_cast<const float4*>(reinterpret_cast<const float*>(upd_src(e)) + int64_t(i) * sld + jb);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float4 v = gs[k];
        v.x = __fmaf_rn(alpha, w[4 * k], v.x);
        v.y = __fmaf_rn(alpha, w[4 * k + 1], v.y);
        v.z = __fmaf_rn(alpha, w[4 * k + 2], v.z);
        v.w = __fmaf_rn(alpha, w[4 * k + 3], v.w);
        g[k] = v;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      if (jb + c < N) {
        const float old = load_elem(upd_src(e), int64_t(i) * sld + jb + c, e.dtype);
        store_elem(e.out, int64_t(i) * e.ld + jb + c, e.dtype, __fmaf_rn(alpha, w[c], old));
      }
    }
  }
}

// ------------------------------------------------------------------ the kernel

// STAGE selects the epilogue (NS_GRAM, NS_POLY, NS_APPLY, TC_UPDATE); MODE the output
// (OutMode: workspace, the caller's outputs, or the caller's bf16 U). Each instantiation
// holds only its own epilogue code.
template <int STAGE, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads(MODE), 1)
    ns_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr bool FINAL = MODE != OUT_WORKSPACE && MODE != OUT_WORKSPACE_KIND;
  constexpr int NEPI = epi_warps(MODE);   // epilogue warps
  constexpr int SPLIT = NEPI / 4;         // epilogue warps per TMEM quadrant
  constexpr int NST = stages_of(MODE);    // operand ring stages
  constexpr bool STREAM = MODE == OUT_UPDATE_STREAM;
  static_assert(!STREAM || STAGE == TC_UPDATE, "the streamed epilogue is the update's");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* staging = smem + NST * STAGE_BYTES;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + NST * STAGE_BYTES + staging_of(MODE));
  uint64_t* full_bar = bars;                // [NST]  (used in the even CTA)
  uint64_t* empty_bar = bars + NST;         // [NST]
  uint64_t* tfull_bar = bars + 2 * NST;     // [2]
  uint64_t* tempty_bar = tfull_bar + 2;     // [2]       (used in the even CTA)
  uint64_t* drain_bar = tempty_bar + 2;     // [1]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 2 * NEPI);
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
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
  // above may overlap that kernel's last CTAs; nothing below runs before it has completed
  // and its memory is visible. The next launch may start its own set-up from here on.
  // the first tile's parameters reach the constant cache while the previous kernel
  // finishes (they do not depend on it); one warp is enough, the cache is the SM's
  if (warp == 1 && pair < p.total_tiles) {
    Tile t0;
    decode_tile(p, pair, t0);
    const TcGroup& G0 = p.g[t0.g];
    const int touch = t0.row0 ^ t0.col0 ^ t0.nkb ^ G0.M ^ G0.N ^ G0.a_mn ^ G0.b_mn ^
                      G0.a_sym ^ G0.b_sym ^ G0.same_ab ^ G0.slot0 ^ G0.syrk ^ G0.final_out ^
                      int(G0.res_ld) ^ int(G0.out_ld);
    asm volatile("" ::"r"(touch));
  }
  // the producer's lanes fetch the tensor maps while the previous kernel finishes
  if (warp == 0 && lane < 2 * p.ngroups) {
    const TcGroup& G = p.g[lane >> 1];
    const CUtensorMap* map = (lane & 1) ? &G.tmB : &G.tmA;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
  }
  // The epilogue warps read global memory written by earlier kernels, so they wait here.
  // The MMA warp touches only shared memory and TMEM, filled by the producer's loads, and
  // the producer waits just before its first load: both get their first tile's barriers
  // ready while the previous kernel finishes.
  if (warp >= 2) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint64_t limit = p.timeout_ns;
#ifdef MAO_TC_TRACE
  const long long t_cta = clock64();
#endif

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool dep_done = false;  // griddepcontrol.wait passed (before the first global access)
    uint32_t armed = 0, armed_phase = 0;  // leader: stages armed at least once, their phase
    for (int k = 0, tile = pair; ok && tile < p.total_tiles;
         tile = pair_tile(pair, ++k, npairs, p.snake)) {
      Tile t;
      decode_tile(p, tile, t);
      const TcGroup& G = p.g[t.g];
      // lane 0 loads this CTA's A half, lane 1 its B half: one 64 x 128 x 2 box each
      // (K-major: 128 rows, two 64-deep k chunks; MN-major: 128 k rows, two 64-wide chunks)
      const bool is_a = lane == 0;
      const bool active = lane < 2;
      const CUtensorMap* map = is_a ? &G.tmA : &G.tmB;
      const int mn_cfg = is_a ? G.a_mn : G.b_mn;
      const int sym_op = is_a ? G.a_sym : G.b_sym;
      const int op_tile = (is_a ? t.row0 : t.col0) / BN;           // 256-tile of the operand rows
      const uint32_t off = is_a ? 0u : uint32_t(HALF_BYTES);
      const int rc = (is_a ? t.row0 : t.col0) + HALF * int(cta);  // this CTA's M/N range
      // a diagonal tile of a product of a buffer with itself: the B half equals the A half
      const bool share = G.same_ab && t.row0 == t.col0;
      const uint32_t tx_bytes = (share ? 2u : 4u) * uint32_t(HALF_BYTES);  // both CTAs
      for (int kb = 0; kb < t.nkb; ++kb) {
        int okw = 1;
        if (lane == 0) {
#ifdef MAO_TC_TRACE
          const long long tw = clock64();
#endif
          if (!mbar_wait_fast(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, limit)) {
            okw = 0;
          } else if (leader) {
            mbar_expect_tx(smem_u32(&full_bar[stage]), tx_bytes);
            armed |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          }
#ifdef MAO_TC_TRACE
          if (leader) TRACE_ADD(0, tw);
#endif
        }
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        if (!dep_done) {  // the first load reads what the previous kernel wrote
          asm volatile("griddepcontrol.wait;" ::: "memory");
          dep_done = true;
        }
        if (active && !(share && !is_a)) {
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
          const uint32_t dst = smem_u32(ring + stage * STAGE_BYTES) + off;
          const int k0 = kb * BK;
          // below the diagonal of a symmetric operand: transposed view of the upper block
          const bool mn = mn_cfg || (sym_op && op_tile > k0 / BN);
          if (mn) tma_load_4d_pair(dst, map, fb, 0, k0, rc / CHUNK, t.z);
          else tma_load_4d_pair(dst, map, fb, 0, rc, k0 / CHUNK, t.z);
        }
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && STAGE == TC_UPDATE && t.nkb <= 2) {
        // a short product (rank-r update): the epilogue, which will read this CTA's 128 rows
        // of the caller's matrix a tile or two from now, is the bottleneck. Have L2 fetch
        // them while the operands load; issued after the tile's operand loads, which would
        // otherwise queue behind them (the first tile's data came 3 to 4 us later). With
        // longer products the prefetched rows displace operand panels from L2 and the
        // prefetch does not pay.
        const OutEntry oe = p.out_table[G.slot0 + t.z];
        if (oe.flags & OUT_VEC) {
          const int es = oe.dtype == MAO_BF16 ? 2 : 4;
          const uint32_t bytes = uint32_t(min(BN, G.N - t.col0) * es) & ~15u;
          const int r0 = t.row0 + HALF * int(cta);
          // one 128-byte line per lane and step, eight lines (up to 1 KB) per row
          const uint8_t* src = reinterpret_cast<const uint8_t*>(upd_src(oe));
          const int64_t sld = upd_src_ld(oe);
          for (int q = lane; q < HALF * 8; q += 32) {
            const int64_t row = r0 + (q >> 3);
            const uint32_t off = uint32_t(q & 7) * 128u;
            if (row < G.M && off < bytes) prefetch_l2(src + (row * sld + t.col0) * es + off);
          }
        }
      }
    }
    // after an abort, the loads already issued land before the CTA leaves: the leader's full
    // barriers count both CTAs' bytes of every armed stage (bounded waits)
    if (*abort_flag && leader && lane == 0) {
      for (int s = 0; s < NST; ++s)
        if ((armed >> s) & 1u) mbar_drain(smem_u32(&full_bar[s]), (armed_phase >> s) & 1u, 20000000ull);
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
      for (int tile = pair; ok && tile < p.total_tiles;
           tile = pair_tile(pair, ++local, npairs, p.snake)) {
        Tile t;
        decode_tile(p, tile, t);
        const TcGroup& G = p.g[t.g];
        const int acc = local & 1;
        const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
#ifdef MAO_TC_TRACE
        const long long tw0 = clock64();
#endif
        if (!mbar_wait_fast<true>(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        TRACE_ADD(2, tw0);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        const int a_tile = t.row0 / BN, b_tile = t.col0 / BN;
        for (int kb = 0; kb < t.nkb; ++kb) {
          const int k_tile = (kb * BK) / BN;
          const int a_mn = G.a_mn || (G.a_sym && a_tile > k_tile);
          const int b_mn = G.b_mn || (G.b_sym && b_tile > k_tile);
          const uint32_t idesc = instr_desc(a_mn, b_mn);
#ifdef MAO_TC_TRACE
          const long long tw1 = clock64();
#endif
          if (!mbar_wait_fast(smem_u32(&full_bar[stage]), phase, abort_flag, limit)) {
            ok = false;
            break;
          }
          TRACE_ADD(1, tw1);
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[5], 1ull);
          const long long t_issue = clock64();
#endif
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + stage * STAGE_BYTES);
          // a diagonal tile of a buffer times itself reads the A half as B
          const uint32_t b_base = (G.same_ab && t.row0 == t.col0) ? a_base : a_base + HALF_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // K-major: chunk kk/4 holds k 64*(kk/4).., 16 k-elements are 32 bytes along the
            //          swizzled row.
            // MN-major: 16 k-rows are two 1024-byte swizzle atoms; the two 64-wide M/N
            //          chunks are CHUNK_BYTES apart.
            const uint32_t koff = uint32_t(kk >> 2) * CHUNK_BYTES + uint32_t(kk & 3) * 32u;
            const uint64_t ad = a_mn ? smem_desc(a_base + kk * 2048, CHUNK_BYTES, 1024)
                                     : smem_desc(a_base + koff, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc(b_base + kk * 2048, CHUNK_BYTES, 1024)
                                     : smem_desc(b_base + koff, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            issued = true;
          }
          umma_commit_pair(smem_u32(&empty_bar[stage]), 3);
#ifdef MAO_TC_TRACE
          atomicAdd(&g_tc_trace[8], (unsigned long long)(clock64() - t_issue));
#endif
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull_bar[acc]), 3);
      }
      if (!ok && issued) {  // wait for every product in flight before TMEM is freed
        umma_commit_pair(smem_u32(drain_bar), 1);
        mbar_drain(smem_u32(drain_bar), 0u, 1000000000ull);
      }
    }
    __syncwarp();
  } else if (STREAM) {
    // ------------------------------------------- streamed update epilogue (both CTAs)
    // Warp (quad, part) takes blocks part and part + 2 of its tiles: item 2k + e is block
    // part + 2e of the warp's k-th tile. Item j's old values are copied into slot j % 3 of
    // the warp's ring, one commit group per item (empty for a block that is absent or
    // written by the per-row path): items 2k + 2 at the start of tile k, 2k + 3 once item
    // 2k has been written out. So a block's rows are in flight for about a tile before the
    // accumulator is applied to them, and no register holds them meanwhile.
    const int quad = warp & 3;
    const int part = (warp - 2) / 4;
    uint8_t* slots = staging + (warp - 2) * STREAM_SLOTS * EP_BYTES;
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty_bar[0]), 0),
                                       mapa_shared(smem_u32(&tempty_bar[1]), 0)};
    auto fill = [&](const Tile& t, const OutEntry& e, int pos, int j) {
      const TcGroup& G = p.g[t.g];
      const int nb = min(BN / 64, (G.N - t.col0 + 63) / 64);
      const int b = part + SPLIT * pos;
      const int jb = t.col0 + 64 * b;
      if (b < nb && upd_block_vec(e, jb, G.N))
        slot_fill(e, slots + (j % STREAM_SLOTS) * EP_BYTES, t.row0 + HALF * int(cta) + 32 * quad,
                  jb, G.M, lane);
      cp_async_commit();
    };
    int tile = pair;
    Tile tc, tn;
    OutEntry oc, on;
    bool hc = tile < p.total_tiles;
    bool hn = pair_tile(pair, 1, npairs, p.snake) < p.total_tiles;
    if (hc) {
      decode_tile(p, tile, tc);
      oc = p.out_table[p.g[tc.g].slot0 + tc.z];
    }
    if (hn) {
      decode_tile(p, pair_tile(pair, 1, npairs, p.snake), tn);
      on = p.out_table[p.g[tn.g].slot0 + tn.z];
    }
    if (hc) {
      fill(tc, oc, 0, 0);
      fill(tc, oc, 1, 1);
    }
    for (int local = 0; hc; ++local) {
      // the tile after next: its entry is loaded now and used a tile from now
      const int tile2 = pair_tile(pair, local + 2, npairs, p.snake);
      const bool h2 = tile2 < p.total_tiles;
      Tile t2;
      OutEntry o2;
      if (h2) {
        decode_tile(p, tile2, t2);
        o2 = p.out_table[p.g[t2.g].slot0 + t2.z];
      }
      const int j0 = 2 * local;
      if (hn) fill(tn, on, 0, j0 + 2);
      else cp_async_commit();
      const TcGroup& G = p.g[tc.g];
      const int acc = local & 1;
      const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
      const bool scaled = p.scale != nullptr;
      const float s = scaled ? p.scale[G.slot0 + tc.z] : 1.0f;
      const int i0 = tc.row0 + HALF * int(cta) + 32 * quad;
      const int nb = min(BN / 64, (G.N - tc.col0 + 63) / 64);
#ifdef MAO_TC_TRACE
      const long long tw2 = clock64();
#endif
      // every lane waits; the warp goes on only if all of them saw the accumulator (the
      // TMEM loads below are warp-wide), so a lane that timed out stops the whole warp
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_fast(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, limit)))
        break;
      tc_fence_after();
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) TRACE_ADD(3, tw2);
      const long long tb = clock64();
#endif
      const uint32_t trow = tmem_base + (uint32_t(32 * quad) << 16) + uint32_t(acc * BN);
      bool vec[2] = {false, false};
#pragma unroll
      for (int pos = 0; pos < 2; ++pos) {
        const int b = part + SPLIT * pos;
        if (pos == 0) cp_async_wait<2>();
        else cp_async_wait<1>();
        __syncwarp();
        if (b >= nb) continue;
        const int jb = tc.col0 + 64 * b;
        float w[64];
        tmem_ld64(trow + uint32_t(64 * b), w);
        if (scaled) {
#pragma unroll
          for (int c = 0; c < 64; ++c) w[c] *= s;
        }
        vec[pos] = upd_block_vec(oc, jb, G.N);
        if (vec[pos]) slot_apply(slots + ((j0 + pos) % STREAM_SLOTS) * EP_BYTES, lane, w, G.alpha);
        else update_final(oc, i0, jb, G.M, G.N, lane, w, G.alpha);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
      // the new rows leave after the accumulator has been released
      if (vec[0]) slot_store(oc, slots + (j0 % STREAM_SLOTS) * EP_BYTES, i0, tc.col0 + 64 * part,
                             G.M, lane);
      __syncwarp();
      if (hn) fill(tn, on, 1, j0 + 3);
      else cp_async_commit();
      if (vec[1]) slot_store(oc, slots + ((j0 + 1) % STREAM_SLOTS) * EP_BYTES, i0,
                             tc.col0 + 64 * (part + SPLIT), G.M, lane);
      __syncwarp();
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) {
        TRACE_ADD(4, tb);
        if (warp == 2) atomicAdd(&g_tc_trace[6], 1ull);
      }
#endif
      tile = pair_tile(pair, local + 1, npairs, p.snake);
      tc = tn;
      oc = on;
      hc = hn;
      tn = t2;
      on = o2;
      hn = h2;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;              // TMEM lanes 32*quad .. 32*quad+31 = this warp's rows
    const int part = (warp - 2) / 4;        // which of the quadrant's SPLIT warps
    // staging: OUT_CALLER, four warps with two buffers each; otherwise eight warps with one
    uint8_t* buf[2] = {staging + (warp - 2) * (2 / SPLIT) * EP_BYTES,
                       staging + ((warp - 2) * (2 / SPLIT) + (SPLIT == 1 ? 1 : 0)) * EP_BYTES};
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty_bar[0]), 0),
                                       mapa_shared(smem_u32(&tempty_bar[1]), 0)};
    int local = 0;
    for (int tile = pair; tile < p.total_tiles;
         tile = pair_tile(pair, ++local, npairs, p.snake)) {
      Tile t;
      decode_tile(p, tile, t);
      const TcGroup& G = p.g[t.g];
      const int acc = local & 1;
      const uint32_t acc_phase = uint32_t(local >> 1) & 1u;
      const int slot = G.slot0 + t.z;
      // the Frobenius scale applies in the first iteration only (p.scale is null after)
      const bool scaled = p.scale != nullptr;
      const float s = scaled ? p.scale[slot] : 1.0f;
      OutEntry oe;
      if (FINAL) oe = p.out_table[slot];
      const int i0 = t.row0 + HALF * int(cta) + 32 * quad;
      const int i = i0 + lane;
      // blocks of 64 columns of the tile (the last one reaches into the zero padding);
      // this warp takes blocks part, part + SPLIT, ...
      const int nb = min(BN / 64, (G.N - t.col0 + 63) / 64);
      // NS_POLY: this warp's residual rows (A) are fetched while the accumulator is still
      // being produced (at most two blocks per warp per tile)
      uint4 res0[8], res1[8];
      if (STAGE == NS_POLY) {
        const __nv_bfloat16* res =
            reinterpret_cast<const __nv_bfloat16*>(G.res) + int64_t(t.z) * G.res_mstride;
        static_assert(STAGE != NS_POLY || SPLIT == 2, "residual registers cover two blocks");
        if (part < nb) load_res_block(res, G.res_ld, i0, t.col0 + 64 * part, G.M, lane, res0);
        if (part + SPLIT < nb)
          load_res_block(res, G.res_ld, i0, t.col0 + 64 * (part + SPLIT), G.M, lane, res1);
      }
      // TC_UPDATE: the old values of the caller's rows, likewise
      if (STAGE == TC_UPDATE) {
        static_assert(STAGE != TC_UPDATE || SPLIT == 2, "prefetch registers cover two blocks");
        const int jb0 = t.col0 + 64 * part, jb1 = t.col0 + 64 * (part + SPLIT);
        if (part < nb && upd_block_vec(oe, jb0, G.N)) upd_load(oe, i0, jb0, G.M, lane, res0);
        if (part + SPLIT < nb && upd_block_vec(oe, jb1, G.N)) upd_load(oe, i0, jb1, G.M, lane, res1);
      }
#ifdef MAO_TC_TRACE
      const long long tw2 = clock64();
#endif
      // every lane waits; the warp goes on only if all of them saw the accumulator (the
      // TMEM loads below are warp-wide), so a lane that timed out stops the whole warp
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_fast(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, limit)))
        break;
      tc_fence_after();
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) TRACE_ADD(3, tw2);
      const long long tb = clock64();
#endif
      const uint32_t trow = tmem_base + (uint32_t(32 * quad) << 16) + uint32_t(acc * BN);
      // unrolled so that the residual registers are selected at compile time
#pragma unroll
      for (int nth = 0; nth < 4 / SPLIT; ++nth) {
        const int b = part + SPLIT * nth;
        if (b >= nb) break;
        const int jb = t.col0 + 64 * b;
        uint8_t* S = buf[nth & 1];
        float w[64];
        tmem_ld64(trow + uint32_t(64 * b), w);
        if (STAGE == NS_GRAM) {
          if (scaled) {
            const float alpha = s * s;
#pragma unroll
            for (int c = 0; c < 64; ++c) w[c] *= alpha;
          }
        } else if (STAGE == NS_POLY) {
          // B' = c (A A) + b A, plus a on the diagonal
          // the staging buffer must have been read by this warp's previous bulk store
          uint4(&r)[8] = nth == 0 ? res0 : res1;
          if (lane == 0) bulk_wait_read();
          __syncwarp();
          res_rows(S, lane, r);
#pragma unroll
          for (int c = 0; c < 64; ++c) w[c] = __fmaf_rn(p.c, w[c], p.b * res_elem(r, c));
          if (i0 < jb + 64 && jb < i0 + 32) {  // the block meets the diagonal
#pragma unroll
            for (int c = 0; c < 64; ++c) w[c] += (jb + c == i) ? p.a : 0.0f;
          }
        } else if ((STAGE == NS_APPLY || STAGE == TC_UPDATE) && scaled) {
          // (TC_UPDATE: the last product of a one-step Newton–Schulz updating W in place)
#pragma unroll
          for (int c = 0; c < 64; ++c) w[c] *= s;
        }
        if (STAGE == TC_UPDATE) {
          if (upd_block_vec(oe, jb, G.N)) upd_apply(S, lane, w, G.alpha, nth == 0 ? res0 : res1);
          else update_final(oe, i0, jb, G.M, G.N, lane, w, G.alpha);
        } else if (MODE == OUT_CALLER_BF16) {
          stage_rows(S, lane, w);
          __syncwarp();
          store_rows(S, reinterpret_cast<__nv_bfloat16*>(oe.out), oe.ld, i0, jb, G.M, G.N, lane);
          __syncwarp();
        } else if (FINAL) {
          store_final(oe, S, i0, jb, G.M, G.N, G.orig_cols, lane, w);
        } else if (MODE == OUT_WORKSPACE_KIND &&
                   (G.out_kind == OUTK_F32 || G.out_kind == OUTK_F32_COLSQ)) {
          // fp32: two 32-column halves, each through the staging buffer (32 rows of 128
          // bytes) and a bulk store; with OUTK_F32_COLSQ lane c then sums the squares of
          // column c of the staged rows (one row per step: conflict-free reads)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (lane == 0) bulk_wait_read();
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(S + srow(lane, k)) =
                  make_float4(w[32 * h + 4 * k], w[32 * h + 4 * k + 1], w[32 * h + 4 * k + 2],
                              w[32 * h + 4 * k + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&G.tmOR, smem_u32(S), jb + 32 * h, i0, t.z);
              bulk_commit();
            }
            if (G.out_kind == OUTK_F32_COLSQ) {
              const int col = jb + 32 * h + lane;
              float sq = 0.0f;
#pragma unroll 8
              for (int rr = 0; rr < 32; ++rr) {
                const float x = *reinterpret_cast<const float*>(S + srow(rr, lane >> 2) + 4 * (lane & 3));
                sq = __fmaf_rn(x, x, sq);
              }
              if (col < G.colsq_ld && i0 < G.M)
                G.colsq[int64_t(t.z) * G.colsq_mstride + int64_t(i0 >> 5) * G.colsq_ld + col] = sq;
            }
            __syncwarp();
          }
        } else if (MODE == OUT_WORKSPACE_KIND && G.out_kind == OUTK_PARTS) {
          // the bf16 parts hi | hi | mid | lo of the fp32 values, out_ld / 4 columns apart,
          // each through the staging buffer and bulk stores (the buffer must have been read
          // by the warp's previous bulk store before it is rewritten)
          const int pl = int(G.out_ld >> 2);
#pragma unroll 1
          for (int q = 0; q < 3; ++q) {
            if (lane == 0) bulk_wait_read();
            __syncwarp();
            stage_rows(S, lane, w);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (q == 0) tma_store_3d(&G.tmOR, smem_u32(S), jb, i0, t.z);
              tma_store_3d(&G.tmOR, smem_u32(S), jb + (q + 1) * pl, i0, t.z);
              bulk_commit();
            }
            __syncwarp();
            if (q < 2) {
#pragma unroll
              for (int c = 0; c < 64; ++c) w[c] -= __bfloat162float(__float2bfloat16_rn(w[c]));
            }
          }
        } else {
          // workspace outputs cover the zero-padded row: the bulk store writes the whole
          // 64-column block (its padding columns hold zeros). The single staging buffer
          // must have been read by this warp's previous bulk store.
          if (lane == 0) bulk_wait_read();
          __syncwarp();
          stage_rows(S, lane, w);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&G.tmOR, smem_u32(S), jb, i0, t.z);
            bulk_commit();
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
      // TC_UPDATE: the rows are written after the accumulator is released, so that the
      // arrive (a release at cluster scope) does not wait for these stores
      if (STAGE == TC_UPDATE) {
        const int jb0 = t.col0 + 64 * part, jb1 = t.col0 + 64 * (part + SPLIT);
        if (part < nb && upd_block_vec(oe, jb0, G.N)) upd_store(oe, i0, jb0, G.M, lane, res0);
        if (part + SPLIT < nb && upd_block_vec(oe, jb1, G.N)) upd_store(oe, i0, jb1, G.M, lane, res1);
      }
#ifdef MAO_TC_TRACE
      if (lane == 0 && leader) {
        TRACE_ADD(4, tb);
        if (warp == 2) atomicAdd(&g_tc_trace[6], 1ull);
      }
#endif
    }
    if (lane == 0) bulk_wait_all();  // stores complete before the CTA leaves
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
#ifdef MAO_TC_TRACE
  if (threadIdx.x == 0 && leader) TRACE_ADD(7, t_cta);
#endif
  if (*abort_flag) {  // an aborted CTA also gives the peer's copies in flight 50 us to land
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 50000ull) {
    }
  }
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

mao_status tc_encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                         int64_t count, int64_t cols) {
  auto fn = encode_fn();
  if (cols < 0) cols = ld;
  if (!fn || ld % CHUNK != 0 || cols % CHUNK != 0 || cols > ld) return MAO_ERR_UNSUPPORTED;
  // dims: 64 columns of a chunk, rows, column chunks (128 bytes apart; the first cols / 64
  // of each row, chunks past them read as zeros), matrices
  const cuuint64_t dims[4] = {cuuint64_t(CHUNK), cuuint64_t(rows), cuuint64_t(cols / CHUNK),
                              cuuint64_t(count)};
  const cuuint64_t strides[3] = {cuuint64_t(ld) * 2, cuuint64_t(CHUNK) * 2,
                                 cuuint64_t(rows) * cuuint64_t(ld) * 2};
  const cuuint32_t box[4] = {CHUNK, HALF, 2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MAO_OK : MAO_ERR_UNSUPPORTED;
}

mao_status tc_encode_store_map_f32(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                                   int64_t count) {
  auto fn = encode_fn();
  if (!fn) return MAO_ERR_UNSUPPORTED;
  const cuuint64_t dims[3] = {cuuint64_t(ld), cuuint64_t(rows), cuuint64_t(count)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 4, cuuint64_t(rows) * cuuint64_t(ld) * 4};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t box[3] = {32, 32, 1};  // 32 rows of 128 bytes, 128-byte swizzle
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MAO_OK : MAO_ERR_UNSUPPORTED;
}

mao_status tc_encode_store_map(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                               int64_t count) {
  auto fn = encode_fn();
  if (!fn) return MAO_ERR_UNSUPPORTED;
  const cuuint64_t dims[3] = {cuuint64_t(ld), cuuint64_t(rows), cuuint64_t(count)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2, cuuint64_t(rows) * cuuint64_t(ld) * 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t box[3] = {64, 32, 1};  // 32 rows of 128 bytes, 128-byte swizzle
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MAO_OK : MAO_ERR_UNSUPPORTED;
}

mao_status tc_gemm_launch(const TcParams& p, cudaStream_t stream) {
  if (p.total_tiles <= 0) return MAO_OK;
  using Kernel = void (*)(TcParams);
  const Kernel kernels[8] = {
      ns_tc_kernel<NS_GRAM, OUT_WORKSPACE>, ns_tc_kernel<NS_POLY, OUT_WORKSPACE>,
      ns_tc_kernel<NS_APPLY, OUT_WORKSPACE>, ns_tc_kernel<NS_APPLY, OUT_CALLER>,
      ns_tc_kernel<TC_UPDATE, OUT_CALLER_BF16>, ns_tc_kernel<NS_APPLY, OUT_CALLER_BF16>,
      ns_tc_kernel<TC_UPDATE, OUT_UPDATE_STREAM>, ns_tc_kernel<NS_APPLY, OUT_WORKSPACE_KIND>};
  static std::once_flag attr_once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MAO_ERR_CUDA;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    for (int i = 0; i < 8; ++i) {
      const size_t bytes = smem_of(i == 6 ? OUT_UPDATE_STREAM : OUT_WORKSPACE);
      const cudaError_t e =
          cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
      if (e != cudaSuccess) attr_err = e;
    }
  });
  if (attr_err != cudaSuccess) return MAO_ERR_CUDA;
  // every group of one launch is either final or not (the last iteration's product); the
  // rank-k update always writes the caller's matrices
  const bool final_out = p.g[0].final_out != 0 || p.stage == TC_UPDATE;
  if (p.stage < NS_GRAM || p.stage > TC_UPDATE || (final_out && p.stage < NS_APPLY))
    return MAO_ERR_INVALID_ARG;
  // the update writes through its own paths with eight epilogue warps: streamed through
  // shared memory when every product is short (the epilogue bounds it), else from registers
  bool short_k = true;
  for (int g = 0; g < p.ngroups; ++g) short_k = short_k && p.g[g].K <= STREAM_MAX_KB * BK;
  const int mode = !final_out ? OUT_WORKSPACE
                   : p.stage == TC_UPDATE && short_k ? OUT_UPDATE_STREAM
                   : p.stage == TC_UPDATE ||
                           (p.stage == NS_APPLY && p.out_mode == OUT_CALLER_BF16)
                       ? OUT_CALLER_BF16
                       : OUT_CALLER;
  bool kind = false;  // a workspace output other than bf16
  for (int g = 0; g < p.ngroups; ++g) kind = kind || p.g[g].out_kind != OUTK_BF16;
  if (kind && (final_out || p.stage != NS_APPLY)) return MAO_ERR_INVALID_ARG;
  const Kernel k = kind ? kernels[7]
                   : mode == OUT_UPDATE_STREAM ? kernels[6]
                   : p.stage == TC_UPDATE  ? kernels[4]
                   : mode == OUT_CALLER_BF16 ? kernels[5]
                   : kernels[final_out ? 3 : p.stage - NS_GRAM];
  const int pairs = p.total_tiles < num_sms() / 2 ? p.total_tiles : num_sms() / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * pairs));
  cfg.blockDim = dim3(unsigned(threads(mode)));
  cfg.dynamicSmemBytes = smem_of(mode);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  profile_before_launch(stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, k, p);
  count_launch();
  profile_after_launch(stream);
  return err == cudaSuccess ? cuda_status(cudaGetLastError()) : MAO_ERR_CUDA;
}

#ifdef MAO_TC_TRACE
extern "C" int mao_debug_tc_trace(unsigned long long* out, int reset) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(out, g_tc_trace, sizeof(unsigned long long) * 16) != cudaSuccess)
    return -1;
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
