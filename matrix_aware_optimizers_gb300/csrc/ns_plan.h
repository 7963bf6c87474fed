// Newton–Schulz execution plan: shape groups, workspace layout and the launch parameters
// of the grouped product kernels (tensor-core bf16 path and fp32 FFMA path).
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "internal.h"
#include "mao.h"

namespace mao {

// Matrices of one original shape R x C. The iteration runs on X (m x n, m <= n): X is the
// matrix itself when R <= C ("wide") and its transpose when R > C ("tall"); in both cases
// the workspace holds the matrix in its original row-major R x C orientation.
struct NsGroupPlan {
  int64_t R, C, m, n;
  bool tall;
  int32_t count;       // matrices in the group
  int32_t slot0;       // first slot (slots are numbered group by group)
  int64_t ldx;         // workspace row stride of X (elements, multiple of 8)
  int64_t lda;         // workspace row stride of A and B (elements, multiple of 8)
  size_t off_x[2];     // ping/pong X buffers [count][R][ldx]
  size_t off_a, off_b; // [count][m][lda]
};

struct NsPlan {
  int es = 2;                          // workspace element size (2: bf16, 4: fp32)
  std::vector<NsGroupPlan> groups;
  std::vector<int32_t> slot_of;        // input index -> slot
  std::vector<int32_t> input_of;       // slot -> input index
  std::vector<int64_t> partial_begin;  // slot -> first partial-sum index
  int64_t n_partials = 0;
  size_t off_out_table = 0, off_scale = 0, off_prange = 0, off_partials = 0;
  size_t total = 0;
};

// Stage-in work decomposition (shared by the plan and the stage-in launch).
constexpr int kStageThreads = 256;
constexpr int kStageUnitsPerBlock = kStageThreads * 4;  // 8 elements per unit

bool make_ns_plan(const mao_mat* X, int32_t batch, int32_t compute, NsPlan& plan);

// --------------------------------------------------------- tensor-core product kernel

namespace tc {
// Tiles of TILE_M x BN outputs are computed by a pair of CTAs (a cluster of two on two SMs,
// tcgen05 cta_group::2): each CTA holds 128 rows of the A operand tile and 128 columns of
// the B operand tile per pipeline stage and receives 128 output rows in its TMEM.
constexpr int TILE_M = 256;      // output rows per tile
constexpr int BN = 256;          // output columns per tile
constexpr int BK = 128;          // reduction depth per pipeline stage
constexpr int HALF = 128;        // rows (A) / columns (B) of the operand tile held per CTA
constexpr int CHUNK = 64;        // columns of one 128-byte swizzle row (bf16)
constexpr int LD_ALIGN = 64;     // workspace rows are padded (with zeros) to CHUNK columns
#ifndef MAO_TC_STAGES
#define MAO_TC_STAGES 3
#endif
constexpr int STAGES = MAO_TC_STAGES;
// Every operand half is one TMA box of 64 x 128 x 2 (two 64-column chunks of 128 rows,
// chunk c at byte offset c * CHUNK_BYTES): 32 KB.
constexpr int CHUNK_BYTES = HALF * CHUNK * 2;     // 16 KB
constexpr int HALF_BYTES = 2 * CHUNK_BYTES;       // 32 KB
constexpr int STAGE_BYTES = 2 * HALF_BYTES;       // A half + B half
// Output modes of a launch: the workspace (bulk tensor stores), the caller's outputs in any
// form (U in fp32 or bf16 with any row stride, packed signs, in-place updates), or the
// caller's bf16 U with 16-byte aligned rows and no signs.
// OUT_UPDATE_STREAM: the in-place update of a short product (rank-k update), whose
// epilogue streams the caller's rows through shared memory (below).
// OUT_WORKSPACE_KIND: workspace outputs of another kind than bf16 (TcGroup::out_kind: bf16
// parts or fp32), kept out of the Newton–Schulz instantiations.
enum OutMode : int {
  OUT_WORKSPACE = 0,
  OUT_CALLER = 1,
  OUT_CALLER_BF16 = 2,
  OUT_UPDATE_STREAM = 3,
  OUT_WORKSPACE_KIND = 4
};
// Epilogue warps: two per 32-lane TMEM quadrant (eight), each taking every other 64-column
// block of the tile, with one staging buffer each; OUT_CALLER uses one warp per quadrant
// (four) with two staging buffers each (its general output code needs more registers).
// Both layouts stage 32 KB.
constexpr int epi_warps(int mode) { return mode == OUT_CALLER ? 4 : 8; }
// warp 0 TMA, warp 1 MMA, then the epilogue warps
constexpr int threads(int mode) { return 64 + 32 * epi_warps(mode); }
constexpr int TMEM_COLS = 512;   // two 256-column fp32 accumulators
// Epilogue staging: 32 x 64 bf16 row-major blocks (128-byte rows, 16-byte chunks XOR-
// swizzled by row).
constexpr int EP_BYTES = 32 * 64 * 2;             // 4 KB
constexpr int STAGING_BYTES = 8 * EP_BYTES;       // 32 KB
// OUT_UPDATE_STREAM: a 2-stage operand ring (a short product keeps the tensor cores busy
// with one tile's operands in flight), and per epilogue warp a ring of STREAM_SLOTS staging
// blocks into which the warp copies the old values of its next blocks (cp.async) while it
// works on the current ones.
constexpr int STREAM_STAGES = 2;
constexpr int STREAM_SLOTS = 3;
constexpr int STREAM_MAX_KB = 2;                  // products of at most 2 k-blocks (K <= 256)
constexpr int stages_of(int mode) { return mode == OUT_UPDATE_STREAM ? STREAM_STAGES : STAGES; }
constexpr int staging_of(int mode) {
  return mode == OUT_UPDATE_STREAM ? 8 * STREAM_SLOTS * EP_BYTES : STAGING_BYTES;
}
constexpr size_t smem_of(int mode) {
  return 1024 /*align*/ + size_t(stages_of(mode)) * STAGE_BYTES + size_t(staging_of(mode)) +
         256 /*barriers*/;
}
constexpr int MAX_GROUPS = 8;
constexpr size_t SMEM_BYTES = smem_of(OUT_WORKSPACE);
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
static_assert(smem_of(OUT_UPDATE_STREAM) <= 232448, "shared memory budget of one CTA");
}  // namespace tc

enum NsStage : int32_t { NS_GRAM = 1, NS_POLY = 2, NS_APPLY = 3 };
enum OutKind : int32_t { OUTK_BF16 = 0, OUTK_PARTS = 1, OUTK_F32 = 2, OUTK_F32_COLSQ = 3 };
// Products of the same kernel outside Newton–Schulz: an in-place rank-k update of the
// caller's matrix, out <- out + a * (A B^T), written through the slot's OutEntry.
constexpr int32_t TC_UPDATE = 4;

struct TcGroup {
  CUtensorMap tmA;          // operand A source (4-D: 64 columns, rows, column chunk, matrix)
  CUtensorMap tmB;          // operand B source
  CUtensorMap tmOR;         // workspace output, 64 x 32 blocks, 128-byte swizzle (bulk stores)
  void* out;                // product output buffer base (workspace), bf16
  const void* res;          // residual buffer base (A for NS_POLY, X for NS_APPLY), bf16
  int64_t out_mstride, res_mstride;  // elements between matrices
  int64_t out_ld, res_ld;            // elements between rows
  int32_t M, N, K;          // product shape: (M x K) . (K x N)
  int32_t count, slot0;
  int32_t a_mn, b_mn;       // operand stored MN-major (1) or K-major (0)
  int32_t a_sym, b_sym;     // operand is a symmetric product stored as its upper and
                            // diagonal 256-tiles: blocks below the diagonal are read
                            // through the transposed (MN-major) view of the upper block
  int32_t syrk;             // symmetric result: only upper and diagonal tiles computed
  int32_t same_ab;          // A and B operands are the same buffer, layout and view: a
                            // diagonal tile loads one half and multiplies it by itself
  int32_t tiles_m, tiles_n, tiles_per_mat, tile_begin;
  int32_t final_out;        // last NS_APPLY: write U / signs through the slot's OutEntry
  int32_t out_kind;         // workspace output (NS_APPLY): OUTK_BF16; OUTK_PARTS, the bf16
                            // parts hi | hi | mid | lo of the fp32 values (hi = bf16(x),
                            // mid = bf16(x - hi), lo = bf16(x - hi - mid)), out_ld / 4
                            // columns apart; OUTK_F32 (tmOR from tc_encode_store_map_f32);
                            // OUTK_F32_COLSQ: fp32, and the column sums of squares of every
                            // 32 rows into colsq (below)
  int32_t orig_cols;        // C of the original matrix (sign-bit indexing)
  float alpha;              // TC_UPDATE: out <- out + alpha (A B^T) for this group's outputs
  float* colsq;             // OUTK_F32_COLSQ: [count] x colsq_mstride floats; the sum of
                            // squares of column j over rows 32 b .. 32 b + 31 at
                            // b * colsq_ld + j (j < colsq_ld)
  int64_t colsq_mstride;
  int32_t colsq_ld;
};

struct TcParams {
  TcGroup g[tc::MAX_GROUPS];
  int32_t ngroups, total_tiles, stage;
  int32_t out_mode;              // final launches: OUT_CALLER or OUT_CALLER_BF16
  float a, b, c;                 // this iteration's coefficients
  const float* scale;            // first iteration: per-slot 1/(||X||_F + eps); else null
  const OutEntry* out_table;     // per-slot final outputs
  unsigned long long timeout_ns; // bound of every barrier wait
  int32_t snake;                 // deal tiles in alternating rounds (see pair_tile)
};

// Operand map of [count][rows][ld] bf16 buffers (ld a multiple of 64); cols (a multiple of
// 64, at most ld; -1 for ld) limits the columns read, later ones load as zeros.
mao_status tc_encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                         int64_t count, int64_t cols = -1);
// Bulk-store map of a workspace output buffer [count][rows][ld] bf16 (64 x 32 blocks).
// fp32 [count][rows][ld] for bulk stores of 32 x 32 blocks (128-byte swizzle)
mao_status tc_encode_store_map_f32(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                                   int64_t count);
mao_status tc_encode_store_map(CUtensorMap* map, const void* base, int64_t rows, int64_t ld,
                               int64_t count);
mao_status tc_gemm_launch(const TcParams& p, cudaStream_t stream);

}  // namespace mao
