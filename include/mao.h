/*
 * mao.h — C ABI of the GB300 (sm_103a) Muon / Sign-Muon optimizer step.
 *
 * One optimizer step, for one weight matrix or a batch of them, is
 *
 *   momentum      M <- mu*M + G                                  muon_momentum_update
 *   polar factor  U ~ polar(M) by Newton–Schulz                   ns_orthogonalize
 *   sign + pack   S = sign(U), one bit per entry                  sign_pack_bits (or fused
 *                                                                 into ns_orthogonalize)
 *   vote          S_bar = sign(sum_m S^(m)) over W_n workers      majority_vote_packed
 *   update        W <- W - eta*S_bar  (Sign-Muon)                 apply_update
 *                 W <- W - eta*U      (Muon)
 *
 * and the two variants the Sign-Muon page describes beside that path:
 *
 *   int8 signs    S = sign(U) as int8 +-1                         sign_int8
 *   SUM + vote    sum_m S^(m) in int8, then S_bar = sign(sum)     majority_vote_int8
 *   polar step    U_bar ~ polar(S_bar) (optional, local)          ns_orthogonalize with an
 *                                                                 MAO_I8 / MAO_SIGN1 input
 *   update        W <- W - eta*U_bar                              apply_update (U form)
 *
 * and the blockwise orthogonalisation of the Megatron page    ns_orthogonalize_blockwise
 * and one step of Dion, the low-rank orthonormal optimizer    dion_step
 *
 * Sources, cited by page title and section:
 *   [SignMuon] "Resumo Técnico: SignMuon: Otimização Distribuída de Muon com Eficiência de
 *              Comunicação" (gist.science, paper 2605.16311), §2 "Metodologia: Sign-Muon".
 *   [Megatron] "NVIDIA MegatronによるLLM学習高速化へ向けた新世代オプティマイザの高度化"
 *              (news.ainew.jp), sections "分散ニュートン・シュルツ" and "SYRK と融合された all-reduce".
 *   [Dion]     "대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습"
 *              (dsdanielpark.github.io), ablation section (heavy-ball momentum form).
 *
 * Conventions shared by every call
 *   - Matrices are row-major: element (i, j) of a mao_mat lives at data + (i*ld + j)*elem_size.
 *     data is a DEVICE pointer, aligned to the element size (16-byte alignment with ld a
 *     multiple of 8 selects the vectorised paths; other layouts take element-wise paths).
 *   - Descriptor arrays (const mao_mat*, pointer arrays) are HOST arrays of `batch` entries,
 *     read during the call only. The caller owns all memory; the library allocates none.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every call only enqueues
 *     work on it and returns; results are ready when the stream reaches that point.
 *   - Argument errors are reported synchronously and enqueue nothing. A failed launch
 *     returns MAO_ERR_CUDA. A device-side wait that ran out of time (MAO_ERR_TIMEOUT) is
 *     reported by mao_sync_status().
 *   - No C++ exception crosses this boundary. Calls are thread-safe per stream.
 *   - Packed sign buffers: entry k of the row-major R x C matrix (k = i*C + j, original
 *     orientation) is bit k%32 of uint32 word k/32, least significant bit first; bit 1
 *     encodes +1 and bit 0 encodes -1 (u < 0). ceil(R*C/32) words; padding bits are 0.
 */
#ifndef MAO_H
#define MAO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mao_status {
  MAO_OK = 0,
  MAO_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum */
  MAO_ERR_UNSUPPORTED = 2,  /* valid request the library cannot serve (device, limits) */
  MAO_ERR_MISALIGNED = 3,   /* pointer not aligned to its element size / workspace to 256 B */
  MAO_ERR_WORKSPACE = 4,    /* workspace smaller than ns_workspace_bytes() */
  MAO_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  MAO_ERR_TIMEOUT = 6,      /* a device-side wait gave up (reported by mao_sync_status) */
  MAO_ERR_NUMERIC = 7       /* a factorisation met a non-positive pivot (mao_sync_status) */
} mao_status;

/*
 * MAO_F32 and MAO_BF16 are storage types of every matrix argument. MAO_I8 and MAO_SIGN1 are
 * accepted only as the INPUT of ns_orthogonalize / ns_orthogonalize_noalloc (the optional
 * polar step on an aggregated sign matrix):
 *   MAO_I8     int8 values, element (i, j) at (int8_t*)data + i*ld + j (any int8 value is
 *              taken as its integer; a sign matrix holds -1 / +1);
 *   MAO_SIGN1  packed signs in the layout of the header comment (uint32 words, 4-byte
 *              aligned data); ld must equal cols; bit 1 -> +1.0, bit 0 -> -1.0.
 */
typedef enum mao_dtype { MAO_F32 = 0, MAO_BF16 = 1, MAO_I8 = 2, MAO_SIGN1 = 3 } mao_dtype;

typedef struct mao_mat {
  void* data;     /* device pointer, row-major */
  int64_t rows;   /* R >= 1 */
  int64_t cols;   /* C >= 1 */
  int64_t ld;     /* elements between consecutive row starts, ld >= cols */
  int32_t dtype;  /* mao_dtype */
  int32_t reserved; /* must be 0 */
} mao_mat;

/* Version of this ABI (bumped on any incompatible change). */
int32_t mao_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* mao_status_string(mao_status status);

/*
 * Momentum of each worker / matrix ([SignMuon] §2 "Fluxo Algorítmico", step 1: each worker
 * updates its local momentum; the form M <- mu*M + G is the heavy-ball form of the [Dion]
 * ablation section).
 *   M[b]  in/out, f32 or bf16; G[b] in, f32 or bf16, same rows/cols as M[b].
 *   Per element: m = fmaf(mu, m, g) in fp32, then round-to-nearest-even to M's dtype.
 *   batch >= 1 matrices of any shapes. M and G must not overlap.
 */
mao_status muon_momentum_update(const mao_mat* M, const mao_mat* G, int32_t batch, float mu,
                                void* stream);

/*
 * Bytes of device workspace ns_orthogonalize needs for this batch (its descriptors' shapes
 * and the compute dtype; pointers are not read). Returns 0 for invalid arguments.
 */
size_t ns_workspace_bytes(const mao_mat* X, int32_t batch, int32_t compute_dtype);

/*
 * Newton–Schulz orthogonalisation toward the polar factor ([SignMuon] §2 "Mecanismo Central"
 * item 1; three matrix products per iteration as [Megatron] "分散ニュートン・シュルツ" counts them;
 * the first two are symmetric rank-k products as in [Megatron] "SYRK と融合された all-reduce").
 *
 * For each matrix (m = min(R,C), X taken as in[b] or its transpose so that X is m x n):
 *   X_0 = X / (||X||_F + eps)
 *   for k in 0..steps-1:  A = X X^T;  B = b_k A + c_k A A;  X = a_k X + B X
 *   U = X (transposed back when R > C; no transposed copy is ever materialised).
 *   The last two products are evaluated as B' = a_k I + b_k A + c_k A A, X = B' X (the same
 *   polynomial; the bf16 operand B' then rounds a + ... instead of the smaller-margin B).
 *
 *   in[b]        f32 or bf16 input (the momentum); read only. For the optional polar step
 *                on an aggregated sign matrix ([SignMuon] §2 step 5) the input may also be
 *                MAO_I8 or MAO_SIGN1 (see mao_dtype); it is converted exactly on staging.
 *   out[b]       f32 or bf16 output U, same rows/cols as in[b]; out[b].data may be NULL when
 *                sign_bits is given (signs only). out may alias in (in-place).
 *   steps        1..64 iterations.
 *   coeffs       HOST array of (a, b, c) triples: 3 floats when coeff_stride == 0 (same
 *                triple every iteration) or steps*3 floats when coeff_stride == 3.
 *   eps          added to the Frobenius norm (1e-7 is the usual value).
 *   compute      MAO_BF16: operands stored in bf16, products on tcgen05 tensor cores with
 *                fp32 accumulation and fp32 epilogue arithmetic;
 *                MAO_F32: fp32 storage and fp32 FFMA products (accuracy path).
 *   sign_bits    NULL, or HOST array of `batch` device pointers (each may be NULL): the
 *                packed signs of the final U (layout in the header comment), written by the
 *                last product's epilogue from the fp32 value before any output rounding.
 *   workspace    device buffer of >= ns_workspace_bytes(in, batch, compute) bytes, 256-byte
 *                aligned; clobbered. Calls sharing a workspace must be stream-ordered.
 */
mao_status ns_orthogonalize(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                            const float* coeffs, int32_t coeff_stride, float eps,
                            int32_t compute, uint32_t* const* sign_bits, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * One whole Muon step in one call ([Dion] ablation section for the heavy-ball momentum
 * M <- mu M + G; [SignMuon] §2 "Fluxo Algorítmico" for the polar factor of the momentum and
 * the update W <- W - eta U): for each matrix
 *   M <- fmaf(mu, M, G)       rounded to M's dtype, written back
 *   U  = Newton–Schulz(M)     exactly as ns_orthogonalize with compute = MAO_BF16
 *   W' = fmaf(-lr, U, W)      rounded to W's dtype, into W_out[b] (or W[b] in place)
 * The momentum is applied by the staging pass that copies M into the workspace, and the
 * last product updates W in its epilogue: U is never stored, and W's update uses U's fp32
 * values (the composed calls round U to the caller's U buffer first).
 *
 *   W, M, G      f32 or bf16 matrices of equal shape per entry (M and G also as for
 *                muon_momentum_update); M is updated in place. No two of W[b], M[b], G[b]
 *                may overlap.
 *   W_out        NULL (W is updated in place) or HOST array of `batch` matrices of W's shape
 *                and dtype receiving W' (W then is only read; W_out[b] may alias W[b] but
 *                must not overlap M[b] or G[b]). Double-buffered weights avoid a copy when
 *                the previous W' is still being read elsewhere.
 *   mu, lr       finite; steps, coeffs, coeff_stride, eps as for ns_orthogonalize.
 *   compute      MAO_BF16 (tensor cores) only; MAO_F32 returns MAO_ERR_UNSUPPORTED.
 *   workspace    >= ns_workspace_bytes(M, batch, MAO_BF16) bytes, 256-byte aligned.
 * Errors: as ns_orthogonalize (argument checks before any launch; device time-outs through
 * mao_sync_status).
 */
mao_status muon_step(const mao_mat* W, const mao_mat* M, const mao_mat* G, const mao_mat* W_out,
                     int32_t batch, float mu, float lr, int32_t steps, const float* coeffs,
                     int32_t coeff_stride, float eps, int32_t compute, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * muon_step with the data on the host: the gradients come in from host memory and the new
 * weights go back to it, all enqueued on `stream` (no counterpart on the pages: the
 * end-to-end form of the step a training loop calls with host-resident gradients). In
 * stream order:
 *   1. g_bytes bytes from g_host (host, preferably pinned) to g_dev (device);
 *   2. if wait_event is not NULL, the stream waits for it (a cudaEvent_t);
 *   3. muon_step(W, M, G, W_out, ...) exactly as that call (G must lie in g_dev's bytes);
 *   4. if record_event is not NULL, it is recorded (a cudaEvent_t);
 *   5. w_bytes bytes from w_dev (device: the new weights, W_out's or W's storage) to w_host.
 * Byte counts may be 0 (that copy is skipped). The events let a caller alternate two streams
 * so that one step's copies overlap its neighbours' compute: step k waits for the event
 * step k-1 recorded after its compute. Argument errors of muon_step, and a NULL buffer for a
 * non-zero copy, are reported before anything is enqueued; a failed copy returns
 * MAO_ERR_CUDA.
 */
mao_status muon_step_host(const mao_mat* W, const mao_mat* M, const mao_mat* G,
                          const mao_mat* W_out, int32_t batch, float mu, float lr, int32_t steps,
                          const float* coeffs, int32_t coeff_stride, float eps, int32_t compute,
                          void* workspace, size_t workspace_bytes, const void* g_host,
                          void* g_dev, size_t g_bytes, void* w_host, const void* w_dev,
                          size_t w_bytes, void* stream, void* wait_event, void* record_event);

/*
 * One whole Sign-Muon step in one call ([SignMuon] §2 "Fluxo Algorítmico", steps 1-4, with
 * the 1-bit all-gather variant; on one GPU the W_n workers' packed buffers already sit in
 * the all-gather layout): the four stages of the calls above, in order on `stream`,
 *   M^(m) <- fmaf(mu, M^(m), G^(m))          muon_momentum_update over the workers
 *   U^(m)  = Newton–Schulz(M^(m))             ns_orthogonalize, signs only: the packed
 *                                             signs of U^(m) into words + m*stride
 *   vote   = sign(sum_m S^(m)), ties -> +1    majority_vote_packed
 *   W     <- fmaf(-lr, vote, W)               apply_update with the vote
 * with the results of those calls bit for bit (U itself is not stored). Launches: with fp32
 * compute and workers small enough for the one-launch Newton–Schulz kernel, the momentum
 * runs inside that launch; with bf16 compute it runs in the pass that stages the workers'
 * M for the tensor-core products; the vote and the update of W are always one pass. So two
 * launches for small fp32 workers, the Newton–Schulz launches plus one with bf16 compute,
 * plus two otherwise.
 *   W          one f32 or bf16 matrix (in/out).
 *   M, G       HOST arrays of n_workers matrices of W's shape (M in/out, G read).
 *   words      device, n_workers rows of worker_stride_words >= ceil(R*C/32) uint32 words
 *              (written); vote: device, ceil(R*C/32) words (written).
 *   steps, coeffs, coeff_stride, eps, compute as ns_orthogonalize; workspace of at least
 *   ns_workspace_bytes(M, n_workers, compute) bytes, 256-byte aligned.
 * Errors: as the four calls (argument checks before any launch).
 */
mao_status sign_muon_step(const mao_mat* W, const mao_mat* M, const mao_mat* G,
                          int32_t n_workers, uint32_t* words, int64_t worker_stride_words,
                          uint32_t* vote, float mu, float lr, int32_t steps, const float* coeffs,
                          int32_t coeff_stride, float eps, int32_t compute, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Size of the scratch area ns_orthogonalize_noalloc uses (16 MiB per device). */
#define MAO_NOALLOC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/* MAO_NOALLOC_WORKSPACE_BYTES as compiled into the library (no counterpart on the pages):
 * the largest ns_workspace_bytes() that ns_orthogonalize_noalloc accepts. */
size_t ns_noalloc_workspace_bytes(void);

/*
 * ns_orthogonalize without a workspace argument. The pages have no counterpart of this
 * call: it exists for callers that cannot call cudaMalloc, such as code inside a host
 * framework that owns all device memory through its own pool, or a latency-critical loop
 * that must not pay cudaMalloc's implicit device synchronisation. Such a caller passes only
 * inputs and outputs; the scratch is one static 16 MiB device array inside this library.
 *
 *   Arguments, results and errors are those of ns_orthogonalize (same kernels, same math).
 *   Limit: the batch must satisfy ns_workspace_bytes(in, batch, compute) <=
 *     MAO_NOALLOC_WORKSPACE_BYTES (for example one 1024 x 1024 or one 768 x 3072 matrix in
 *     bf16); larger requests return MAO_ERR_WORKSPACE before any device work.
 *   Memory: allocates nothing. Every GPU that loads this library holds the 16 MiB array
 *     until the process exits, whether or not the call is used.
 *   Set-up: every call made outside stream capture looks up the array's device address
 *     (cudaGetSymbolAddress) with the current device, so a call after cudaDeviceReset or
 *     in another context finds the array where that context loaded it. A call made while
 *     its stream is being captured reuses the address of the last call on that device, so
 *     make the first call on each device (and the first after a device reset) outside any
 *     capture; a captured call without such an earlier call returns MAO_ERR_UNSUPPORTED.
 *   Sharing: all calls on a device use the same array, which keeps the last call's
 *     contents (nothing in it needs to start at zero). Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on it: order them on one stream or with
 *     events.
 */
mao_status ns_orthogonalize_noalloc(const mao_mat* in, const mao_mat* out, int32_t batch,
                                    int32_t steps, const float* coeffs, int32_t coeff_stride,
                                    float eps, int32_t compute, uint32_t* const* sign_bits,
                                    void* stream);

/*
 * Blockwise Newton–Schulz ([Megatron] "分散モード", blockwise paragraph: each rank
 * orthogonalises only the block of the momentum it owns; no communication, and not the
 * orthogonalisation of the whole matrix).
 *
 * Each matrix is cut into a grid of block_rows x block_cols blocks (the last block row and
 * column take what is left); every block is orthogonalised on its own exactly as
 * ns_orthogonalize would orthogonalise that block alone (its own Frobenius norm, its own
 * orientation), and written to the same place of out[b]. Blocks of equal shape run as one
 * group; the blocks are read and written in place through strides (no copies).
 *   in[b]        f32, bf16 or MAO_I8 (not MAO_SIGN1); out[b] f32 or bf16, same shape.
 *   block_rows, block_cols   >= 1; at most 2^20 blocks per call (else MAO_ERR_UNSUPPORTED).
 *   Other arguments as ns_orthogonalize (no sign output); workspace of at least
 *   ns_blockwise_workspace_bytes(in, batch, block_rows, block_cols, compute) bytes.
 */
size_t ns_blockwise_workspace_bytes(const mao_mat* X, int32_t batch, int64_t block_rows,
                                    int64_t block_cols, int32_t compute_dtype);
mao_status ns_orthogonalize_blockwise(const mao_mat* in, const mao_mat* out, int32_t batch,
                                      int64_t block_rows, int64_t block_cols, int32_t steps,
                                      const float* coeffs, int32_t coeff_stride, float eps,
                                      int32_t compute, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * Entrywise sign and 1-bit packing ([SignMuon] §2 step 2 "Extração de Sinal" and step 3,
 * all-gather variant: one bit per entry).
 *   U     f32 or bf16 matrix (read). bits: device array of ceil(R*C/32) words (written).
 *   sign(u) = -1 (bit 0) if u < 0, else +1 (bit 1): +0, -0 and NaN give +1.
 */
mao_status sign_pack_bits(const mao_mat* U, uint32_t* bits, void* stream);

/*
 * Majority vote over W_n workers' packed sign buffers ([SignMuon] §2 step 4: the vote
 * S_bar = sign(sum_m S^(m)) computed locally after the all-gather of packed buffers).
 *   bits           device, worker m's words start at bits + m*worker_stride_words
 *                  (the all-gather result layout; worker_stride_words >= ceil(nbits/32)).
 *   n_workers      1..65535.   nbits  entries per worker (>= 1).
 *   vote           device, ceil(nbits/32) words written: bit = 1 where the number of +1
 *                  signs is >= the number of -1 signs (a tie gives +1); padding bits 0.
 */
mao_status majority_vote_packed(const uint32_t* bits, int32_t n_workers,
                                int64_t worker_stride_words, int64_t nbits, uint32_t* vote,
                                void* stream);

/*
 * Entrywise sign as int8 ([SignMuon] §2 step 2, for the all-reduce variant of step 3 and the
 * "8 bits with int8" payload of "Eficiência de Comunicação").
 *   U     f32 or bf16 matrix (read).
 *   s     device array of R*C int8 (written), row-major packed: s[i*C + j] = -1 if
 *         U(i, j) < 0, else +1 (+0, -0 and NaN give +1).
 */
mao_status sign_int8(const mao_mat* U, int8_t* s, void* stream);

/*
 * Integer SUM of W_n workers' int8 sign buffers followed by the local threshold
 * ([SignMuon] §2 step 3, all-reduce variant, and step 4: S_bar = sign(sum_m S^(m))).
 * On one GPU the workers' buffers sit side by side and the SUM all-reduce is the reduction
 * over them; its result is the int8 buffer an int8 SUM all-reduce would leave on every
 * worker.
 *   s              device, worker m's n entries start at s + m*worker_stride (bytes,
 *                  worker_stride >= n). Entries are expected in {-1, +1}; any int8 values
 *                  are summed as integers.
 *   n_workers      1..127 (the int8 sum of +-1 signs is then exact).
 *   n              entries per worker (>= 1).
 *   sum            NULL or device array of n int8: sum_m S^(m) (wraps modulo 256 only if
 *                  the entries are not +-1).
 *   s_bar          NULL or device array of n int8: +1 where sum >= 0 (a tie gives +1), else -1.
 *   vote           NULL or device array of ceil(n/32) words: S_bar packed (header layout).
 *   At least one of sum, s_bar, vote must be non-NULL. Outputs must not overlap s.
 */
mao_status majority_vote_int8(const int8_t* s, int32_t n_workers, int64_t worker_stride,
                              int64_t n, int8_t* sum, int8_t* s_bar, uint32_t* vote,
                              void* stream);

/*
 * Parameter update ([SignMuon] §2 step 4: W_{t+1} = W_t - eta_t * S_bar_t).
 *   W[b]     in/out, f32 or bf16.
 *   Exactly one of:
 *     vote   HOST array of `batch` device pointers to packed signs of W[b]'s shape
 *            (Sign-Muon: D = +1 for bit 1, -1 for bit 0);
 *     U      HOST array of `batch` matrices of W[b]'s shape, f32 or bf16 (Muon: D = U).
 *   Per element: w = fmaf(-lr, d, w) in fp32, then round-to-nearest-even to W's dtype.
 */
mao_status apply_update(const mao_mat* W, const uint32_t* const* vote, const mao_mat* U,
                        int32_t batch, float lr, void* stream);

/*
 * One Dion step ([Dion] "대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습",
 * algorithm section) for `batch` parameter matrices of any shapes m x n (grouped by shape
 * inside the call) and one rank r:
 *
 *   B = M + G;  P = orthonormalise(B Q);  R = B^T P
 *   M <- B - (1 - mu) P R^T;  Q <- ColumnNormalize(R);  X <- X - lr P Q^T
 *
 * orthonormalise gives the Q factor of the thin QR of B Q with a positive triangular
 * diagonal, computed as Cholesky QR applied twice: the Gram matrix P^T P and the product
 * with L^-1 on the tensor cores from bf16 parts of their fp32 factors (fp32 accumulation;
 * the Gram to about fp32 accuracy, the product to about 2^-17), the Cholesky factor L and
 * its inverse in fp32 on CUDA cores; ColumnNormalize divides each
 * column by its Euclidean norm (a zero column stays zero).
 *   X[b], M[b]  in/out, f32 or bf16, m x n;  G[b] in, f32 or bf16, m x n.
 *   Q[b]        in/out, f32, n x r (any ld): the previous right factor in, the new one out.
 *   X_out       NULL (X is updated in place), or HOST array of `batch` matrices of X[b]'s
 *               shape and dtype receiving X - lr P Q^T; X is then only read. X_out[b] may
 *               be X[b] itself (same data and ld: in place) and must not overlap it
 *               otherwise. Lets a caller read back one step's X while the next step runs.
 *   P_out       NULL, or HOST array of `batch` device pointers (each may be NULL): the
 *               final P, m x r fp32, row stride r.
 *   rank        1..256, at most min(m, n) of every matrix; batch <= 65535.
 *   compute     MAO_BF16 only: B, Q, P and R enter the dense products (B Q, B^T P,
 *               P R^T / P Q^T) as bf16 with fp32 accumulation on tcgen05 tensor cores; the
 *               two products of Cholesky QR use bf16 parts of fp32 factors as above; the
 *               rest (staging sums, Cholesky, norms, the updates' arithmetic) is fp32.
 *   workspace   >= dion_workspace_bytes(X, batch, rank) bytes, 256-byte aligned.
 *   Errors: MAO_ERR_INVALID_ARG for mismatched shapes of X, M, G, Q, X_out (or X_out's
 *   dtype differing from X's) or a bad rank;
 *   B Q without full column rank (a non-positive Cholesky pivot) is reported by
 *   mao_sync_status() as MAO_ERR_NUMERIC (the pivot is replaced by 1e-30).
 */
size_t dion_workspace_bytes(const mao_mat* X, int32_t batch, int32_t rank);
mao_status dion_step(const mao_mat* X, const mao_mat* M, const mao_mat* G, const mao_mat* Q,
                     const mao_mat* X_out, float* const* P_out, int32_t batch, int32_t rank,
                     float mu, float lr, int32_t compute, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Bound of every device-side wait of the tensor-core kernels (default 4 s), used by launches
 * enqueued after the call; process-wide. A wait that runs past it makes the kernel stop
 * early (its outputs are then incomplete) and mao_sync_status() report MAO_ERR_TIMEOUT.
 * 0 makes every wait that does not complete at once give up: the way to exercise that path
 * without a GPU fault. mao_get_wait_limit returns the current bound.
 */
void mao_set_wait_limit(uint64_t ns);
uint64_t mao_get_wait_limit(void);

/*
 * Synchronise `stream`, then read and clear the device-side error words that kernels set
 * when a bounded wait gives up or a factorisation meets a non-positive pivot. Returns
 * MAO_OK, MAO_ERR_TIMEOUT, MAO_ERR_NUMERIC or MAO_ERR_CUDA.
 */
mao_status mao_sync_status(void* stream);

/*
 * Measurement support (no counterpart on the pages; used by benchmarks).
 *
 * mao_launch_count: number of kernels this library has launched in this process.
 *
 * mao_profile_begin: from now on, every launch of the tensor-core product kernel (three
 *   per Newton–Schulz iteration, four per Dion step), of the Dion CUDA-core kernels and of
 *   the one-launch fp32 Newton–Schulz of small matrices is
 *   bracketed by a pair of CUDA events recorded on the launch's stream, for up to
 *   max_launches launches (1..1<<20). Creates the events
 *   (host-side driver objects, no device memory). Not thread-safe: one profiling session
 *   per process. Returns MAO_ERR_INVALID_ARG for a bad count, MAO_ERR_CUDA on failure.
 *
 * mao_profile_end: stops recording, synchronises the recorded events, writes the elapsed
 *   milliseconds of up to max_out recorded launches into ms_out (host array, may be NULL
 *   when max_out is 0), destroys the events and returns the number of launches recorded
 *   (negative on a CUDA error).
 *
 * mao_profile_end_tagged: as mao_profile_end, and also writes one tag per recorded launch
 *   into tags_out (host array of max_out entries, may be NULL): MAO_PROF_TC for the
 *   tensor-core product kernel, otherwise the MAO_PROF_DION_* value of the Dion kernel or
 *   MAO_PROF_NS_SMALL.
 */
enum {
  MAO_PROF_TC = 0,
  MAO_PROF_DION_SETUP = 1,     /* device table of the slots */
  MAO_PROF_DION_STAGE = 2,     /* B = M + G and its bf16 copy; bf16 copy of Q_prev */
  MAO_PROF_DION_GRAM = 3,      /* P^T P assembled from its tensor-core parts (the products are MAO_PROF_TC) */
  MAO_PROF_DION_CHOL = 4,      /* Cholesky factor and its inverse */
  MAO_PROF_DION_SPLIT = 5,     /* unused: P's bf16 parts and the final P are written by the products (MAO_PROF_TC) */
  MAO_PROF_DION_NORM = 6,      /* column norms of R, Q = ColumnNormalize(R) */
  MAO_PROF_NS_SMALL = 7        /* the one-launch fp32 Newton–Schulz of small matrices */
};
int64_t mao_launch_count(void);
mao_status mao_profile_begin(int32_t max_launches);
/*
 * mao_profile_span_begin / mao_profile_span_end: as mao_profile_begin / mao_profile_end, but
 *   one event pair per Newton–Schulz call on the tensor cores (ns_orthogonalize, muon_step,
 *   ...): recorded before its first product launch and after its last, so the products keep
 *   overlapping one another's set-up (programmatic dependent launch) while they are timed.
 *   Returns the number of recorded spans and their durations in milliseconds. Independent of
 *   the per-launch session; use one of them at a time.
 */
mao_status mao_profile_span_begin(int32_t max_spans);
int32_t mao_profile_span_end(float* ms_out, int32_t max_out);
int32_t mao_profile_end(float* ms_out, int32_t max_out);
int32_t mao_profile_end_tagged(float* ms_out, int32_t* tags_out, int32_t max_out);

#ifdef __cplusplus
}
#endif

#endif /* MAO_H */
