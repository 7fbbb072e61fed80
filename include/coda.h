/*
 * coda.h - C ABI of libcoda: BF16 GEMMs on GB300 (sm_103a) whose output tile
 * is transformed on chip by a small epilogue program before it is stored, plus
 * the light auxiliary reductions that combine the epilogues' tile partials,
 * and an unfused comparison path (plain GEMM + separate element-wise kernels).
 *
 * The method is CODA, "Rewriting Transformer Blocks as GEMM-Epilogue Programs".
 * Citations name the page and the passage:
 *   "CODA note"  the papernotes.org note on the paper (method section, Key
 *                designs 1-4; kernel and block speedup tables);
 *   "pith page"  the pith.science page on arXiv 2605.19269 (figure captions,
 *                Appendix A.1).
 *
 * Conventions for every entry point
 *   - Tensors are device pointers, allocated and owned by the caller. The
 *     library never allocates, frees or retains caller memory. Its own device
 *     memory is the status word, the static array of coda_block_fwd_noalloc
 *     and one stream-K workspace per stream that uses the split
 *     (coda_set_stream_k), each kept until the process exits.
 *   - bf16 tensors are passed as coda_bf16 (uint16_t bit patterns), row-major
 *     and contiguous unless a leading dimension (in elements) is given.
 *     Statistics are fp32, labels int32. Weights are [K, N] row-major.
 *   - Base pointers of bf16 tensors and vectors and of fp32 tables must be
 *     16-byte aligned; every row stride must be a multiple of 16 bytes
 *     (8 bf16 elements). fp32 / int32 vectors (r, s, lse, labels, partials)
 *     need only natural alignment.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and do not synchronise. Outputs must not alias inputs
 *     unless stated.
 *   - The fused GEMMs and the auxiliary reductions are launched with
 *     programmatic stream serialization: each kernel may be scheduled while
 *     the previous kernel on the stream finishes, and waits for it
 *     (griddepcontrol.wait) before touching memory, so stream order holds as
 *     for plain launches. A caller's own kernel launched after a coda call
 *     with the same attribute must likewise wait (cudaGridDependencySynchronize)
 *     before reading the call's outputs.
 *   - A dimension of 0 makes the call a no-op that returns CODA_OK (an empty
 *     contraction, K = 0, gives a zero accumulator and the epilogue still runs).
 *   - Return value: CODA_OK, or a negative CODA_ERR_*; coda_last_error()
 *     describes the last failure on the calling thread. Argument errors are
 *     detected on the host before anything is launched.
 *   - Kernels never trap. Each mbarrier wait inside them is bounded; a wait
 *     that runs out sets CODA_DEVST_TIMEOUT in the device status word and the
 *     kernel returns early. Out-of-range labels set CODA_DEVST_BAD_LABEL. A
 *     split tile whose arrival word could not be updated (see coda_set_stream_k)
 *     sets CODA_DEVST_SPLIT and is left unwritten.
 *     Read (and clear) the word with coda_device_status().
 *   - A checked build of the same library (libcoda_checked.so, compiled with
 *     CODA_CHECKED=1) tests the index of every direct global load and store
 *     of the fused epilogues (row statistics, tile partials, per-row vectors,
 *     RoPE tables) against the tensor's extent before the access; an index
 *     outside sets CODA_DEVST_BOUNDS and the access is skipped. TMA loads and
 *     stores are bounded by their tensor maps in both builds.
 *   - Per-device state (the status word's address, kernel attributes, the
 *     cluster count, the no-allocation scratch's address) is set up by the
 *     first call on a device and kept for the life of the process: it assumes
 *     one CUDA context per device. After cudaDeviceReset() on a device, do not
 *     use the library on that device again in the same process.
 */
#ifndef CODA_H_
#define CODA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CODA_OK 0
#define CODA_ERR_INVALID (-1)     /* null pointer, misalignment, bad dimension   */
#define CODA_ERR_UNSUPPORTED (-2) /* shape granularity not supported, not sm_103 */
#define CODA_ERR_CUDA (-3)        /* a CUDA runtime / driver call failed         */
#define CODA_ERR_TIMEOUT (-4)     /* device status word reported a timeout       */

#define CODA_DEVST_TIMEOUT 1   /* a bounded in-kernel wait ran out            */
#define CODA_DEVST_BAD_LABEL 2 /* a cross-entropy label was outside [0, V)    */
#define CODA_DEVST_BOUNDS 4    /* checked build only: an epilogue's direct global access fell outside its tensor */
#define CODA_DEVST_SPLIT 8     /* a split tile's arrival word could not be updated; that tile is not written */

typedef uint16_t coda_bf16;
typedef void* coda_stream_t;

/* ------------------------------------------------------------------ runtime */

/* Thread-local text of the last error (empty string if none). */
const char* coda_last_error(void);

/* Make `device` current, check it is compute capability 10.3 (GB300), cache its
 * SM count. Other calls do this lazily for the current device. */
int coda_init(int device);

/* Synchronise the current device, return the device status word
 * (CODA_DEVST_* bits, >= 0) and, if `clear` != 0, reset it to 0.
 * Returns CODA_ERR_CUDA if the synchronisation fails. */
int coda_device_status(int clear);

/* Bound on every in-kernel mbarrier wait, in nanoseconds (default 2e9).
 * Values below 1e5 are rejected with CODA_ERR_INVALID. */
int coda_set_wait_timeout_ns(unsigned long long ns);

/* GEMM tile variant for every later launch on this process: 1 = one SM per
 * 128 x 256 tile (tcgen05 cta_group::1); 2 = an SM pair per 256 x 256 tile
 * (cta_group::2, 2-CTA clusters); 0 (default) = the pair whenever M > 128.
 * Results are identical up to fp32 accumulation order. Other values are
 * rejected with CODA_ERR_INVALID. */
int coda_set_cta_group(int g);

/* Stream-K work split for every later launch on this process. A fused GEMM
 * runs as persistent tile loops, one per SM (pair); when the tile count is
 * not a multiple of their number, the last wave leaves most of the GPU idle.
 * With the split on, one wave plus the leftover tiles are instead shared out
 * as equal ranges of k-blocks, run before the remaining whole tiles, so
 * every SM (pair) does the same work; a tile whose k-blocks fall in two
 * ranges is accumulated in two pieces, whose fp32 partials meet in a
 * per-stream workspace, and the piece that finishes second adds them and
 * runs the epilogue.
 *   0 = off: the last wave runs as whole tiles or as 128-column half tiles;
 *   1 = automatic (default): the split where it is expected to be faster
 *       (at least 16 k-blocks of 64, and a last wave that leaves enough of
 *       the GPU idle);
 *   2 = whenever it applies (K >= 1024 and more tiles than one wave).
 * Other values are rejected with CODA_ERR_INVALID.
 * Results stay deterministic: a split tile's accumulator is the fp32 sum of
 * its two pieces, the same whichever finishes first. They differ from the
 * data-parallel schedule's only in fp32 accumulation order.
 * Workspace: a stream's first launch that uses the split allocates its
 * workspace (256 KiB per SM, about 38 MiB on GB300, with cudaMalloc) and
 * zeroes its arrival words on the stream; it is kept until the process
 * exits, one per stream handle (at most 64). Launches made while the stream
 * is being captured into a CUDA graph, and those of coda_block_fwd_noalloc,
 * never use the split, so they allocate nothing and capture no workspace. */
int coda_set_stream_k(int mode);

/* Test hook for the failure-detection path: the next fused-GEMM launch from
 * this process skips the producers' first stage fill, so the MMA issuer's
 * bounded wait on it runs out. The kernel then sets CODA_DEVST_TIMEOUT, stops
 * every role, drains the copies and MMAs it issued, frees TMEM and returns;
 * its outputs are undefined. Use with a short coda_set_wait_timeout_ns(). */
int coda_test_inject_missing_load(void);

/* Number of 128-column blocks of a fused kernel's output for GEMM width N
 * (ceil(N / 128)): the second dimension of every [M, nb] partial buffer.
 * Each partial covers one 128-column block of one row. */
int coda_num_col_tiles(int N);

/* Number of row tiles used by the column partials of coda_gemm_rmsnorm_bwd
 * and coda_unfused_rmsnorm_bwd (ceil(M / 32)). */
int coda_num_row_tiles(int M);

/* ---------------------------------------------------------- plain GEMM (a1)
 * C[M,N] = op(A) op(B), bf16 in, fp32 accumulate on the tensor cores, bf16 out.
 * The fixed mainloop of CODA (CODA note, overall framework) with the identity
 * epilogue. transA = 0: A is [M,K] row-major (lda >= K); transA = 1: A is
 * stored [K,M] row-major (lda >= M) and used transposed. transB = 0: B is
 * [K,N] row-major (ldb >= N); transB = 1: B is stored [N,K] (ldb >= K).
 * ldc >= N. N and K multiples of 8 (with transA, M as well). */
int coda_gemm(int M, int N, int K, const coda_bf16* A, int lda, int transA, const coda_bf16* B, int ldb,
              int transB, coda_bf16* C, int ldc, coda_stream_t stream);

/* --------------------------------------------- GEMM-RMSNorm-GEMM forward (a2-a4)
 * CODA note, Key design 1: RMSNorm(x W0 + z, gamma) W1 = r ((x W0 + z) (.) gamma) W1
 * with r the per-row inverse RMS, applied in the second GEMM's epilogue.
 *
 * coda_gemm_res_rmsprep: first GEMM, epilogue h1 = x W0 + z, h2 = h1 (.) gamma,
 *   psq[i, t] = sum over the columns of block t of h1[i,j]^2 (fp32 h1, before
 *   rounding; the pages' tile partial of the unscaled residual).
 *   x [M,K], W0 [K,N], z [M,N], gamma [N] -> h1, h2 [M,N] bf16,
 *   psq [M, coda_num_col_tiles(N)] fp32. N, K multiples of 8. */
int coda_gemm_res_rmsprep(int M, int N, int K, const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                          const coda_bf16* gamma, coda_bf16* h1_out, coda_bf16* h2_out, float* psq_out,
                          coda_stream_t stream);

/* Auxiliary reduction (pith page, Figures 4 and 5):
 * r[i] = 1 / sqrt(sum_t psq[i,t] / d + eps). psq [M, nb] fp32 -> r [M] fp32. */
int coda_rms_reduce(int M, int nb, int d, const float* psq, float eps, float* r_out, coda_stream_t stream);

/* Second GEMM with the delayed row scale (CODA note, Key design 1):
 * Y[i,j] = r[i] (h2 W1)[i,j]. h2 [M,K], W1 [K,N], r [M] -> Y [M,N] bf16. */
int coda_gemm_rowscale(int M, int N, int K, const coda_bf16* h2, const coda_bf16* W1, const float* r,
                       coda_bf16* Y_out, coda_stream_t stream);

/* ----------------------------------------------------------- SwiGLU (a5, a6)
 * CODA note, Key design 2; pith page, Figure 7: gate and up channels are
 * interleaved (even column = gate G, odd = up U).
 *
 * coda_gemm_swiglu: GU = X Wgu; A[:, f] = silu(GU[:, 2f]) GU[:, 2f+1].
 *   X [M,K], Wgu [K, 2F] -> A [M,F] bf16; gu_out [M,2F] bf16 (the
 *   pre-activation saved for the backward) or NULL. F multiple of 8. */
int coda_gemm_swiglu(int M, int F, int K, const coda_bf16* X, const coda_bf16* Wgu, coda_bf16* A_out,
                     coda_bf16* gu_out, coda_stream_t stream);

/* coda_gemm_swiglu_bwd: dA = dY Wd^T (Wd stored [F, K]: the down-projection
 *   weight), epilogue recomputes sigmoid(G) from gu and emits, interleaved,
 *   dG = dA U s (1 + G (1 - s)), dU = dA G s with s = sigmoid(G).
 *   dY [M,K], Wd [F,K], gu [M,2F] -> dgu [M,2F] bf16. */
int coda_gemm_swiglu_bwd(int M, int F, int K, const coda_bf16* dY, const coda_bf16* Wd, const coda_bf16* gu,
                         coda_bf16* dgu_out, coda_stream_t stream);

/* ------------------------------------------------------------- RoPE (a7, a8)
 * CODA note, Key design 2: rotation of adjacent channel pairs (2i, 2i+1) of
 * each head with pre-broadcast cos/sin vectors.
 *
 * coda_rope_tables: cos_tab[p, i] = cos(p theta^(-2i/head_dim)), sin_tab
 *   likewise, evaluated in fp64 and rounded to fp32; [S, head_dim/2]. */
int coda_rope_tables(int S, int head_dim, double theta, float* cos_out, float* sin_out, coda_stream_t stream);

/* coda_gemm_rope: P = X W; for columns c < rope_cols (the Q and K heads) with
 *   pair i = (c mod head_dim) / 2 at position p = row mod S:
 *   out_e = a_e cos - a_o sin, out_o = a_e sin + a_o cos; columns at or
 *   beyond rope_cols (V) pass through.
 *   X [M,K], W [K,N], cos/sin [S, head_dim/2] fp32 -> out [M,N] bf16.
 *   head_dim a multiple of 32, rope_cols a multiple of head_dim and <= N.
 *   The tables must hold angles linear in the position, cos_tab[p, i] =
 *   cos(p w_i) and sin_tab likewise, as coda_rope_tables writes them: when S
 *   is a multiple of 32 and head_dim <= 128 the kernel forms the values of
 *   positions p0 + l (l < 32, p0 a multiple of 32) by angle addition from
 *   table rows p0 and l. (The same holds for every RoPE epilogue below.) */
int coda_gemm_rope(int M, int N, int K, const coda_bf16* X, const coda_bf16* W, const float* cos_tab,
                   const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out, coda_stream_t stream);

/* coda_gemm_rope_bwd: the same GEMM with the transposed rotation in the
 *   epilogue (duality rule, CODA note, Key design 3): g_e = a_e cos + a_o sin,
 *   g_o = -a_e sin + a_o cos. Arguments as coda_gemm_rope. */
int coda_gemm_rope_bwd(int M, int N, int K, const coda_bf16* A, const coda_bf16* B, const float* cos_tab,
                       const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out,
                       coda_stream_t stream);

/* ---------------------------------------------------- cross-entropy (a9, a10)
 * CODA note, Key design 4 (stateful online log-sum-exp across vocabulary
 * tiles, combined by an auxiliary reduction). Logits L = H W are fp32 in the
 * accumulator and are never stored.
 *
 * coda_gemm_ce_lse: per (row i, 128-column block t): pmax[i,t] = max_j L[i,j],
 *   psum[i,t] = sum_j exp(L[i,j] - pmax[i,t]), parg[i,t] = lowest j attaining
 *   the max (NULL to skip); the block that holds label y_i writes
 *   tgt[i] = L[i, y_i]. H [M,K], W [K,V], labels [M] int32 in [0,V) ->
 *   pmax, psum [M, coda_num_col_tiles(V)] fp32, parg same shape int32, tgt [M].
 *   A label outside [0, V) sets CODA_DEVST_BAD_LABEL and tgt[i] = NaN. */
int coda_gemm_ce_lse(int M, int V, int K, const coda_bf16* H, const coda_bf16* W, const int32_t* labels,
                     float* pmax_out, float* psum_out, int32_t* parg_out, float* tgt_out, coda_stream_t stream);

/* coda_ce_reduce: LSE_i = Mx + ln sum_t psum[i,t] exp(pmax[i,t] - Mx),
 *   Mx = max_t pmax[i,t]; loss_row_i = LSE_i - tgt_i; loss_mean = (1/M) sum_i
 *   loss_row_i (single scalar, NULL to skip); argmax_i from parg (lowest
 *   column among equal maxima; NULL parg or argmax_out to skip). */
int coda_ce_reduce(int M, int nb, const float* pmax, const float* psum, const int32_t* parg, const float* tgt,
                   float* lse_out, float* loss_row_out, float* loss_mean_out, int32_t* argmax_out,
                   coda_stream_t stream);

/* coda_gemm_ce_bwd: recomputes the logits tile and emits
 *   dl[i,j] = grad_scale (exp(L[i,j] - lse_i) - [j == y_i]) in bf16
 *   (grad_scale = g / M for the mean loss). H [M,K], W [K,V], labels [M],
 *   lse [M] -> dl [M,V] bf16. dH = dl W^T and dW = H^T dl are coda_gemm calls. */
int coda_gemm_ce_bwd(int M, int V, int K, const coda_bf16* H, const coda_bf16* W, const int32_t* labels,
                     const float* lse, float grad_scale, coda_bf16* dl_out, coda_stream_t stream);

/* ------------------------------------- GEMM-RMSNorm-GEMM backward (a11, a12)
 * CODA note, Key design 3: s = (1/d) rowsum(dY (.) Y) is formed in the
 * epilogue of the GEMM that produces dY.
 *
 * coda_gemm_rowdot: dY = dO Wn; stores dY (bf16), optionally dYr = r (.)row dY
 *   (bf16; NULL to skip, r may then be NULL), and pdot[i,t] = sum over the
 *   columns of block t of dY[i,j] Y[i,j] (fp32 dY times the stored bf16 Y).
 *   dO [M,K], Wn [K,N], Y [M,N] -> dY, dYr [M,N], pdot [M, coda_num_col_tiles(N)]. */
int coda_gemm_rowdot(int M, int N, int K, const coda_bf16* dO, const coda_bf16* Wn, const coda_bf16* Y,
                     const float* r, coda_bf16* dY_out, coda_bf16* dYr_out, float* pdot_out, coda_stream_t stream);

/* coda_rowdot_reduce: s[i] = sum_t pdot[i,t] / d. */
int coda_rowdot_reduce(int M, int nb, int d, const float* pdot, float* s_out, coda_stream_t stream);

/* coda_gemm_rmsnorm_bwd: G = dY W1^T (W1 stored [d, K] row-major, the forward
 *   weight of the second GEMM); epilogue dh1 = r gamma (.) G - r^2 s h1 and
 *   column partials pdg[b, j] = sum over rows of row tile b of r_i G[i,j] h1[i,j].
 *   dY [M,K], W1 [d,K], h1 [M,d] bf16, gamma [d] bf16, r, s [M] fp32 ->
 *   dh1 [M,d] bf16, pdg [coda_num_row_tiles(M), d] fp32. */
int coda_gemm_rmsnorm_bwd(int M, int d, int K, const coda_bf16* dY, const coda_bf16* W1, const coda_bf16* h1,
                          const coda_bf16* gamma, const float* r, const float* s, coda_bf16* dh1_out,
                          float* pdg_out, coda_stream_t stream);

/* coda_colsum_reduce: dgamma[j] = sum_b pdg[b, j]. pdg [rows, d] -> [d] fp32. */
int coda_colsum_reduce(int rows, int d, const float* pdg, float* dgamma_out, coda_stream_t stream);

/* -------------------------------------------------- unfused comparison path
 * The memory-bound operators CODA removes, as separate HBM-bound kernels that
 * read and write every intermediate (CODA note, research background). Each
 * reads bf16 tensors and writes bf16 tensors; statistics are fp32. */

/* out = a + b, [M,N] bf16 (out may alias a or b). */
int coda_unfused_add(int M, int N, const coda_bf16* a, const coda_bf16* b, coda_bf16* out, coda_stream_t stream);

/* Textbook RMSNorm: r_i = 1/sqrt(mean_j h[i,j]^2 + eps), n = r h (.) gamma.
 * h [M,d], gamma [d] -> n [M,d] bf16, r [M] fp32 (r_out may be NULL). */
int coda_unfused_rmsnorm(int M, int d, const coda_bf16* h, const coda_bf16* gamma, float eps, coda_bf16* n_out,
                         float* r_out, coda_stream_t stream);

/* out = r (.)row x, [M,N] bf16. */
int coda_unfused_rowscale(int M, int N, const coda_bf16* x, const float* r, coda_bf16* out, coda_stream_t stream);

/* A = silu(gu[:, 0::2]) gu[:, 1::2]; gu [M,2F] -> A [M,F]. */
int coda_unfused_swiglu(int M, int F, const coda_bf16* gu, coda_bf16* A_out, coda_stream_t stream);

/* dgu from dA [M,F] and gu [M,2F] (formulas as coda_gemm_swiglu_bwd). */
int coda_unfused_swiglu_bwd(int M, int F, const coda_bf16* dA, const coda_bf16* gu, coda_bf16* dgu_out,
                            coda_stream_t stream);

/* In-place RoPE (forward) / transposed rotation (backward) on x [M,N] bf16. */
int coda_unfused_rope(int M, int N, const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols,
                      coda_bf16* x, coda_stream_t stream);
int coda_unfused_rope_bwd(int M, int N, const float* cos_tab, const float* sin_tab, int S, int head_dim,
                          int rope_cols, coda_bf16* x, coda_stream_t stream);

/* Cross-entropy over materialised bf16 logits [M,V]: lse, loss_row [M],
 * loss_mean (scalar, NULL to skip), argmax [M] (NULL to skip). */
int coda_unfused_ce_fwd(int M, int V, const coda_bf16* logits, const int32_t* labels, float* lse_out,
                        float* loss_row_out, float* loss_mean_out, int32_t* argmax_out, coda_stream_t stream);

/* dl = grad_scale (softmax(logits) - onehot(labels)) from bf16 logits and lse. */
int coda_unfused_ce_bwd(int M, int V, const coda_bf16* logits, const int32_t* labels, const float* lse,
                        float grad_scale, coda_bf16* dl_out, coda_stream_t stream);

/* s_i = (1/d) sum_j dY[i,j] Y[i,j] over bf16 dY, Y [M,N]. */
int coda_unfused_rowdot(int M, int N, int d, const coda_bf16* dY, const coda_bf16* Y, float* s_out,
                        coda_stream_t stream);

/* Textbook RMSNorm backward from G = dL/dn [M,d], h [M,d], gamma [d], r [M]:
 * c_i = (1/d) sum_j G gamma h, dh = r gamma G - r^3 c h; column partials
 * pdg [coda_num_row_tiles(M), d] of r G h (reduce with coda_colsum_reduce). */
int coda_unfused_rmsnorm_bwd(int M, int d, const coda_bf16* G, const coda_bf16* h, const coda_bf16* gamma,
                             const float* r, coda_bf16* dh_out, float* pdg_out, coda_stream_t stream);

/* ------------------------------------------------- FP8 (E4M3) mainloop (f3)
 * CODA note, research background: as FP8 and FP4 GEMMs multiply the tensor
 * throughput, the memory-bound operators around the GEMM take a larger share
 * of the time, which the fused epilogues remove. These entry points run the
 * same epilogue programs as their bf16 twins on an FP8 mainloop (tcgen05
 * kind::f8f6f4, fp32 accumulators in TMEM):
 *   - A [M,K] and B stored [N,K] (both K-major; B in the layout of a linear
 *     layer's weight [out, in]) are E4M3 bytes: 1 sign bit, 4 exponent bits
 *     with bias 7, 3 mantissa bits, no infinities (0x7F / 0xFF are NaN);
 *   - the accumulator is multiplied by alpha, the product of the two operands'
 *     per-tensor scales, before the epilogue program sees it;
 *   - K a multiple of 16 (16-byte rows), N a multiple of 8; base pointers
 *     16-byte aligned. Outputs, statistics, status bits and errors as the bf16
 *     twins. */

/* C[M,N] = alpha A B^T in bf16 (identity epilogue). */
int coda_gemm_fp8(int M, int N, int K, const uint8_t* A, const uint8_t* B, float alpha, coda_bf16* C,
                  coda_stream_t stream);

/* coda_gemm_rope on P = alpha X W^T: X [M,K], W [N,K] E4M3. */
int coda_gemm_rope_fp8(int M, int N, int K, const uint8_t* X, const uint8_t* W, float alpha, const float* cos_tab,
                       const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out, coda_stream_t stream);

/* coda_gemm_swiglu on GU = alpha X Wgu^T: Wgu [2F,K] E4M3, row 2f the gate and
 * row 2f+1 the up projection of output f. gu_out (bf16 [M,2F]) may be NULL. */
int coda_gemm_swiglu_fp8(int M, int F, int K, const uint8_t* X, const uint8_t* Wgu, float alpha, coda_bf16* A_out,
                         coda_bf16* gu_out, coda_stream_t stream);

/* coda_gemm_ce_lse on the logits alpha H W^T: H [M,K], W [V,K] E4M3. */
int coda_gemm_ce_lse_fp8(int M, int V, int K, const uint8_t* H, const uint8_t* W, float alpha, const int32_t* labels,
                         float* pmax_out, float* psum_out, int32_t* parg_out, float* tgt_out, coda_stream_t stream);

/* coda_gemm_ce_bwd on the recomputed logits alpha H W^T. */
int coda_gemm_ce_bwd_fp8(int M, int V, int K, const uint8_t* H, const uint8_t* W, float alpha, const int32_t* labels,
                         const float* lse, float grad_scale, coda_bf16* dl_out, coda_stream_t stream);

/* ------------------------------------------------------ block-level chain (f1)
 * CODA note, block-level ablation: a Transformer block seen as two
 * consecutive GEMM-Residual-RMSNorm-GEMM structures, one on the RoPE path and
 * one on the SwiGLU path, with the light auxiliary reductions and glue. One
 * period of a pre-norm layer stack, the attention core left out (its output O
 * is an input; the attention backward's gradient of the rotated QKV, dQKV, is
 * an input):
 *   RoPE path:   h1 = P Wd + x;  n1 = RMSNorm(h1, gamma1);  QKV = RoPE(n1 Wqkv)
 *   SwiGLU path: h2 = O Wo + h1; n2 = RMSNorm(h2, gamma2);  GU = n2 Wgu;
 *                A = SwiGLU(GU)
 * The backward differentiates L = <dQKV, QKV> + <gh, A Wdn + h2>, where gh is
 * the gradient of the next period's residual output A Wdn + h2 and Wdn [F,d]
 * the next period's down projection. The gradient of the block input P
 * (dh1 Wd^T) is the next-earlier period's SwiGLU-backward GEMM and is not
 * formed here.
 *
 * The four composed kernels below are used by the fused chain; each is also a
 * stand-alone entry point. */

/* coda_gemm_rowscale_rope: out = RoPE(r (.)row (X W)): the delayed row scale
 *   (Key design 1) and the pair rotation (Key design 2) in one epilogue.
 *   X [M,K], W [K,N], r [M] fp32, cos/sin [S, head_dim/2] -> out [M,N] bf16.
 *   Rotation, positions and limits as coda_gemm_rope. */
int coda_gemm_rowscale_rope(int M, int N, int K, const coda_bf16* X, const coda_bf16* W, const float* r,
                            const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols,
                            coda_bf16* out, coda_stream_t stream);

/* coda_gemm_rowscale_swiglu: GU = r (.)row (X Wgu) (the scale precedes the
 *   nonlinearity); A[:, f] = silu(GU[:, 2f]) GU[:, 2f+1]. gu_out (the scaled
 *   pre-activation, [M,2F] bf16) may be NULL. Limits as coda_gemm_swiglu. */
int coda_gemm_rowscale_swiglu(int M, int F, int K, const coda_bf16* X, const coda_bf16* Wgu, const float* r,
                              coda_bf16* A_out, coda_bf16* gu_out, coda_stream_t stream);

/* coda_gemm_swiglu_bwd_rowdot: dA = dY Wd^T (Wd stored [F,K]); the epilogue
 *   forms dGU = SwiGLU'(dA; gu) as coda_gemm_swiglu_bwd, the RMSNorm-backward
 *   row-statistic partials of the rowscale GEMM that produced gu (Key design 3),
 *   pdot[i,t] = sum over the 256 gu columns of dA block t of dGU[i,j] gu[i,j]
 *   (fp32 dGU times the stored bf16 gu), and stores dGUr = r (.)row dGU.
 *   dY [M,K], Wd [F,K], gu [M,2F], r [M] -> dgur [M,2F] bf16,
 *   pdot [M, coda_num_col_tiles(F)] fp32 (s = coda_rowdot_reduce(.., d, ..)). */
int coda_gemm_swiglu_bwd_rowdot(int M, int F, int K, const coda_bf16* dY, const coda_bf16* Wd, const coda_bf16* gu,
                                const float* r, coda_bf16* dgur_out, float* pdot_out, coda_stream_t stream);

/* coda_gemm_rmsnorm_bwd_res: Gr = dYr W1^T (W1 stored [d,K]) on the row-scaled
 *   gradient, so Gr = r (.)row G; epilogue dh = gamma (.) Gr - r^2 s h + dres
 *   (dres: the gradient reaching h through the residual connection) and column
 *   partials pdg[b,j] = sum over the rows of row tile b of Gr[i,j] h[i,j].
 *   dYr [M,K], W1 [d,K], h, dres [M,d] bf16, gamma [d] bf16, r, s [M] ->
 *   dh [M,d] bf16, pdg [coda_num_row_tiles(M), d] fp32. */
int coda_gemm_rmsnorm_bwd_res(int M, int d, int K, const coda_bf16* dYr, const coda_bf16* W1, const coda_bf16* h,
                              const coda_bf16* gamma, const float* r, const float* s, const coda_bf16* dres,
                              coda_bf16* dh_out, float* pdg_out, coda_stream_t stream);

/* coda_rope_bwd_rowdot: the RoPE-path glue of the backward, one pass over the
 *   attention backward's dQKV (no GEMM of the chain produces it):
 *   dYq = RoPE^T(dQKV) (transposed rotation on columns < rope_cols),
 *   s[i] = (1/d) sum_j dQKV[i,j] QKV[i,j] (equal to (1/d) rowsum(dYq (.) Yq)
 *   for the unrotated projection Yq: the rotation is orthogonal), and
 *   dqr = r (.)row dYq. dqkv, qkv [M,N] bf16, r [M], cos/sin [S, head_dim/2]
 *   -> dqr [M,N] bf16, s [M] fp32. head_dim a multiple of 8. HBM-bound. */
int coda_rope_bwd_rowdot(int M, int N, const coda_bf16* dqkv, const coda_bf16* qkv, const float* r,
                         const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols, int d,
                         coda_bf16* dqr_out, float* s_out, coda_stream_t stream);

/* Descriptor of one period of the chain. Sizes: M tokens, d model width, F
 * FFN width (Wgu has 2F interleaved gate/up columns), QKV width 3d with RoPE on
 * columns [0, rope_cols) at position row mod S. All tensors are caller-owned
 * device memory, row-major, bf16 unless marked fp32. The fused and the unfused
 * sequences use the same descriptor; where the meaning differs it says so. */
typedef struct coda_block {
  int M, d, F;
  int head_dim, rope_cols, S;
  float eps;
  const float* cos_tab; /* [S, head_dim/2] fp32 (coda_rope_tables) */
  const float* sin_tab;
  /* forward inputs */
  const coda_bf16* P;      /* [M,F] activation entering the down projection */
  const coda_bf16* x;      /* [M,d] residual stream entering the period */
  const coda_bf16* O;      /* [M,d] attention-core output */
  const coda_bf16* Wd;     /* [F,d] */
  const coda_bf16* gamma1; /* [d] */
  const coda_bf16* Wqkv;   /* [d,3d] */
  const coda_bf16* Wo;     /* [d,d] */
  const coda_bf16* gamma2; /* [d] */
  const coda_bf16* Wgu;    /* [d,2F] */
  /* written by the forward, read by the backward */
  coda_bf16* h1;  /* [M,d] residual stream after the RoPE-path GEMM */
  coda_bf16* h1g; /* [M,d] fused: h1 (.) gamma1; unfused: n1 = RMSNorm(h1) */
  coda_bf16* h2;  /* [M,d] */
  coda_bf16* h2g; /* [M,d] fused: h2 (.) gamma2; unfused: n2 */
  coda_bf16* gu;  /* [M,2F] GU = n2 Wgu (the same tensor on both paths) */
  float* r1;      /* [M] fp32 inverse RMS of h1 */
  float* r2;      /* [M] fp32 */
  /* forward outputs */
  coda_bf16* qkv; /* [M,3d] rotated QKV */
  coda_bf16* a;   /* [M,F] SwiGLU output */
  /* backward inputs */
  coda_bf16* dqkv;       /* [M,3d] gradient of the rotated QKV; the fused backward only reads it, the
                            unfused backward rotates it in place (its RoPE backward works in place) */
  const coda_bf16* gh;   /* [M,d] gradient of the next period's residual output */
  const coda_bf16* Wdn;  /* [F,d] the next period's down projection */
  /* backward outputs */
  coda_bf16* dh1;   /* [M,d] = dL/dx */
  coda_bf16* dh2;   /* [M,d] */
  coda_bf16* dO;    /* [M,d] gradient to the attention core */
  coda_bf16* dWd;   /* [F,d] */
  coda_bf16* dWqkv; /* [d,3d] */
  coda_bf16* dWo;   /* [d,d] */
  coda_bf16* dWgu;  /* [d,2F] */
  float* dgamma1;   /* [d] fp32 */
  float* dgamma2;   /* [d] fp32 */
  /* backward intermediates */
  coda_bf16* dgur; /* [M,2F] fused: r2 (.)row dGU; unfused: dGU */
  coda_bf16* dqr;  /* [M,3d] fused: r1 (.)row RoPE^T(dQKV); unused by the unfused backward (may be NULL) */
  float* s1;       /* [M] fp32 row statistics (fused only) */
  float* s2;
  /* scratch: coda_block_workspace_bytes(M, d, F, unfused) bytes, 256-byte aligned */
  void* workspace;
} coda_block_t;

/* Scratch bytes the chain needs (partials; and for unfused != 0 also the
 * intermediates the unfused sequence materialises). 0 for negative sizes. */
size_t coda_block_workspace_bytes(int M, int d, int F, int unfused);

/* Fused forward: residual + RMS-prep GEMM, coda_rms_reduce,
 * coda_gemm_rowscale_rope; residual + RMS-prep GEMM, coda_rms_reduce,
 * coda_gemm_rowscale_swiglu (GU saved). 6 launches. */
int coda_block_fwd(const coda_block_t* b, coda_stream_t stream);

/* coda_block_fwd_noalloc: the fused forward for callers that cannot allocate
 * device memory: a plugin that its host engine hands only input and output
 * buffers, with no allocator and no workspace; a serving loop that may not
 * call cudaMalloc after start-up, because the call can synchronise the device
 * and take an unbounded time; a process whose memory pool already holds the
 * device's memory. It has no counterpart on the pages (a deployment
 * convenience of this library). It runs the launch sequence of coda_block_fwd but ignores
 * b->workspace: the forward's only scratch, the sum-of-squares partials
 * (M * ceil(d/128) fp32 values), lives in a 4 MiB file-scope device array of
 * the library, one per device. Sizes with M * ceil(d/128) * 4 > 4 MiB return
 * CODA_ERR_UNSUPPORTED (M = 16384 fits up to d = 8192). Two calls whose
 * kernels can overlap on the GPU (calls on different streams, or from threads
 * whose streams are not ordered) race on that array and give undefined
 * results; calls on one stream run in order and are safe. Allocates nothing:
 * its GEMMs never take the stream-K split (coda_set_stream_k), whose
 * per-stream workspace would be allocated, so at sizes where coda_block_fwd
 * splits, the two differ in fp32 accumulation order.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and keeps it for the process; make
 * that first call before any stream capture. */
int coda_block_fwd_noalloc(const coda_block_t* b, coda_stream_t stream);

/* Fused backward (after coda_block_fwd on the same descriptor):
 * coda_gemm_swiglu_bwd_rowdot, coda_rowdot_reduce, coda_gemm_rmsnorm_bwd_res
 * (dres = gh), coda_colsum_reduce, dWgu = h2g^T dgur, dO = dh2 Wo^T,
 * dWo = O^T dh2, coda_rope_bwd_rowdot, coda_gemm_rmsnorm_bwd_res (dres = dh2),
 * coda_colsum_reduce, dWqkv = h1g^T dqr, dWd = P^T dh1. 13 launches. */
int coda_block_bwd(const coda_block_t* b, coda_stream_t stream);

/* Unfused forward: plain GEMMs and the stand-alone kernels (add, RMSNorm,
 * RoPE in place, SwiGLU). 10 launches. */
int coda_block_fwd_unfused(const coda_block_t* b, coda_stream_t stream);

/* Unfused backward (after coda_block_fwd_unfused): plain GEMMs, SwiGLU
 * backward, textbook RMSNorm backward, residual adds, RoPE backward in place
 * on dqkv. 16 launches. */
int coda_block_bwd_unfused(const coda_block_t* b, coda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CODA_H_ */
