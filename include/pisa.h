/*
 * pisa.h - C ABI of the GB300 (sm_103a) piecewise sparse attention library.
 *
 * The library computes the forward pass of PISA, "PISA: Piecewise Sparse
 * Attention Is Wiser for Efficient Diffusion Transformers": per query block,
 * the critical key blocks (the +-band diagonal plus the top-k blocks by pooled
 * score) are attended exactly, and every other key block enters the same
 * softmax numerator and denominator through its block-wise first-order
 * Taylor expansion around the block's key centroid (Section 3.2, Eq. (3)-(6)).
 *
 * Three calls make up the path, in this order:
 *   pisa_block_stats  block means / sums / first-order matrices
 *   pisa_route        critical block list per query block
 *   pisa_forward      the fused exact + approximate attention
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are dense, row-major, innermost (channel) dimension contiguous.
 *   Q, K, V and the output are [heads, n, d]; a batch is folded into `heads`.
 * - Every pointer except `stream` and `dev_status` is a DEVICE pointer to
 *   memory the caller allocated and owns. The library allocates no device
 *   memory and keeps no state between calls; calls are re-entrant. (The one
 *   exception is pisa_forward_hybrid_static, whose scratch is a fixed
 *   device array shared by its calls.)
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call only enqueues work on it and returns without synchronising.
 * - Argument and shape errors are detected on the host before anything is
 *   enqueued and returned as PISA_ERR_INVALID_ARG / PISA_ERR_UNSUPPORTED.
 *   A failed launch returns PISA_ERR_CUDA.
 * - `dev_status` (optional, may be NULL) is a device int32 the caller zeroes
 *   beforehand; a kernel that detects an error at run time (a bounded wait
 *   that expired, a failed bounds check) stores a pisa_status code there and
 *   returns early instead of trapping. Read it after synchronising.
 * - dtype codes: PISA_F32 (IEEE float32) or PISA_BF16 (bfloat16).
 * - The block size is 64 tokens, for queries and keys alike (Section 4.1
 *   "Implementation Details"); head dims 64 and 128.
 *   The last block of a head may hold fewer tokens (n_j = n - 64 (nb - 1)).
 */
#ifndef PISA_H
#define PISA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PISA_OK = 0,
  PISA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or code    */
  PISA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d = 96)      */
  PISA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed  */
  PISA_ERR_TIMEOUT = 4,      /* device: a bounded wait expired              */
  PISA_ERR_DEVICE_CHECK = 5  /* device: a run-time bounds check failed      */
} pisa_status;

typedef enum { PISA_F32 = 0, PISA_BF16 = 1 } pisa_dtype;

/* matrix norm of the block heterogeneity M_j (pisa_block_heterogeneity) */
typedef enum { PISA_NORM_SPECTRAL = 0, PISA_NORM_FROBENIUS = 1 } pisa_norm;

/*
 * pisa_block_stats - per-block statistics of Q, K, V.
 *
 * Source: Section 3.2 "Formulation" (block partition, key centroid
 * kbar_j = mean_n k_{j,n}), Eq. (5) (value block sum Vhat_j = sum_n v_{j,n}),
 * Eq. (6) / Appendix C "Notation" (H_j = sum_n (k_{j,n} - kbar_j)^T v_{j,n}),
 * Figure 4 "Prepare Phase" (block means of the queries, Qbar).
 *
 * q, k, v   [heads, n, d] of `in_dtype`, 16-byte aligned.
 * qbar      [heads, nb, d] float32 out: mean of the n_j queries of block j.
 * kbar      [heads, nb, d] float32 out: mean of the n_j keys of block j.
 * vsum      [heads, nb, d] float32 out: sum of the n_j values of block j.
 * hmat      [heads, nb, d, d] out, element (c, e) = sum_n (k_{j,n,c} -
 *           kbar_{j,c}) v_{j,n,e}; stored as `h_dtype` (F32 or BF16).
 * Each output may be NULL to skip it (at least one must be given); a tensor
 * whose outputs are all NULL is not read. nb = ceil(n / block). Means and
 * sums are accumulated with compensated float32 summation and rounded once.
 * dev_status (optional device int32) receives PISA_ERR_TIMEOUT if a block's
 * rows never arrive in shared memory within the bounded wait (about a
 * second); that block's outputs are then left unwritten. Errors: INVALID_ARG
 * for null inputs, all outputs NULL, misalignment, heads < 1, n < 1,
 * block != 64, unknown dtype; UNSUPPORTED for d not in {64, 128}.
 */
int pisa_block_stats(const void* q, const void* k, const void* v, int in_dtype,
                     int heads, int n, int d, int block,
                     float* qbar, float* kbar, float* vsum,
                     void* hmat, int h_dtype,
                     int32_t* dev_status, void* stream);

/*
 * pisa_global_first_order - the global first-order statistic of the hybrid
 * approximation, Hbar = (1/nb) sum_j H_j, per head.
 *
 * Source: Section 3.3 "Global First-Order Correction", Eq. 10 (Hbar, query
 * independent, precomputed in a single pass); Appendix C "Notation" (H_j
 * centred on the block centroid). Evaluated through the identity
 * sum_j H_j = K^T V - sum_j kbar_j (x) Vhat_j (exact in real arithmetic).
 *
 * k, v      [heads, n, d] of `in_dtype`, 16-byte aligned.
 * kbar, vsum [heads, nb, d] float32 (from pisa_block_stats).
 * hbar      [heads, d, d] float32 out, element (c, e) = key channel c, value
 *           channel e. Overwritten (the call zeroes it on the stream first).
 * bf16 inputs with d = 128 use the tensor cores for K^T V (bf16 products,
 * float32 accumulation); other inputs use float32 CUDA-core arithmetic.
 * The CTAs that share a head form a thread-block cluster and sum their
 * partials in a fixed order: hbar is the same bit for bit on every call.
 * Errors: as pisa_block_stats.
 */
int pisa_global_first_order(const void* k, const void* v, int in_dtype,
                            int heads, int n, int d, int block,
                            const float* kbar, const float* vsum, float* hbar,
                            int32_t* dev_status, void* stream);

/*
 * pisa_route - critical key blocks S_i of every query block.
 *
 * Source: Figure 4 "Prepare Phase" and Algorithm 1 step 2 (top-k selection of
 * key blocks per query block on the pooled score qbar_i . kbar_j, scaled by
 * s); the diagonal band follows the Piecewise-Taylor-Attention README
 * ("Knobs": band=b keeps |i-j| <= b exact).
 *
 * S_i = band(i) U top_k{ j : |i - j| > band } ordered by descending score
 * s * qbar_i . kbar_j, the lower block index winning ties. Because s > 0 the
 * ranking is that of qbar_i . kbar_j, which is evaluated in double-float
 * (about 48-bit) arithmetic from the float32 inputs.
 *
 * qbar, kbar [heads, nb, d] float32 (from pisa_block_stats).
 * scale      s > 0.
 * topk       >= 0 blocks chosen outside the band (all candidates if larger).
 * band       >= 0.
 * idx        [heads, nb, max_sel] int32 out: S_i in ascending order, padded
 *            with -1.
 * cnt        [heads, nb] int32 out: |S_i|.
 * max_sel    row stride of idx; must be >= min(nb, topk + 2 band + 1).
 * Errors: INVALID_ARG for null pointers, nb < 1, heads < 1, topk < 0,
 * band < 0, scale <= 0 or not finite, max_sel too small; UNSUPPORTED for d not
 * in {64, 128} or nb > 16384.
 */
int pisa_route(const float* qbar, const float* kbar, int heads, int nb, int d,
               float scale, int topk, int band,
               int32_t* idx, int32_t* cnt, int max_sel,
               int32_t* dev_status, void* stream);

/*
 * pisa_block_heterogeneity - per-block heterogeneity of the first-order
 * statistics, M_j = || H_j - Hbar ||, the prior of covariance-aware routing.
 *
 * Source: Section 3.3 "Covariance-Aware Block Selection" (M_j, Eq. 11) and
 * Theorem 3.1 (the norm ||.||_2), Appendix D (Eq. 14). H_j is centred on the
 * block's own key centroid (Appendix C "Notation"); Hbar is the global mean
 * from pisa_global_first_order.
 *
 * k, v      [heads, n, d] of `in_dtype`, 16-byte aligned.
 * kbar      [heads, nb, d] float32 (pisa_block_stats).
 * hbar      [heads, d, d] float32 (pisa_global_first_order).
 * norm      PISA_NORM_SPECTRAL: largest singular value (the norm Section 3.3
 *           writes); PISA_NORM_FROBENIUS: root of the sum of squares (the
 *           Piecewise-Taylor-Attention README's router).
 * mnorm     [heads, nb] float32 out, 16-byte aligned.
 * A = H_j - Hbar is formed from the block's tokens (H_j itself is not read or
 * stored): for bf16 inputs with d = 128 on the tensor cores, the centred keys
 * split into three bf16 terms (exact products, float32 accumulation; the
 * Frobenius norm by one persistent CTA per SM that streams the blocks); for
 * other inputs in float32 on the CUDA cores. The spectral norm is the square
 * root of the largest eigenvalue of A^T A by the Lanczos iteration, stopped
 * when the residual of the top Ritz pair is below 1e-7 of it (at most d
 * steps): about float32 precision.
 * Errors: as pisa_block_stats; INVALID_ARG for an unknown norm. A bounded
 * wait of the tensor-core path that runs out writes PISA_ERR_TIMEOUT to
 * *dev_status (when non-NULL) and leaves that block's entry unwritten.
 */
int pisa_block_heterogeneity(const void* k, const void* v, int in_dtype,
                             int heads, int n, int d, int block,
                             const float* kbar, const float* hbar, int norm,
                             float* mnorm, int32_t* dev_status, void* stream);

/*
 * pisa_route_covariance - critical key blocks with the covariance-aware score.
 *
 * Source: Section 3.3 "Covariance-Aware Block Selection", Eq. 11: the pooled
 * logit of key block j gains log(M_j + eps). The softmax of Eq. 11 is monotone
 * and Appendix D's -log(Mbar) is the same for every block, so the selection is
 * the top-k of r_ij = s * qbar_i . kbar_j + log(M_j + eps) outside the band,
 * the lower block index winning ties; the band is added as in pisa_route.
 *
 * mnorm      [heads, nb] float32 (pisa_block_heterogeneity), 16-byte aligned.
 *            An entry that is negative, NaN or infinite is taken as 0 and
 *            reported as PISA_ERR_DEVICE_CHECK in *dev_status.
 * eps        > 0, finite (the pages leave its value open).
 * Other arguments, outputs and errors: as pisa_route. r_ij is evaluated as in
 * pisa_route (float32 screening with a proven bound, double-float scores for
 * the candidates it cannot separate), log(M_j + eps) in double.
 */
int pisa_route_covariance(const float* qbar, const float* kbar, const float* mnorm,
                          float eps, int heads, int nb, int d, float scale,
                          int topk, int band, int32_t* idx, int32_t* cnt,
                          int max_sel, int32_t* dev_status, void* stream);

/*
 * pisa_forward - the piecewise attention output.
 *
 * Source: Section 3.2, Eq. (3)-(6). For query t of query block i, q' = s q_t:
 *   D_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} + sum_{j not in S_i} n_j e^{q'.kbar_j}
 *   N_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} v_{j,n}
 *       + sum_{j not in S_i} e^{q'.kbar_j} (Vhat_j + q' H_j)
 *   o_t = N_t / D_t
 * with one shared running maximum ("Safe-Exp", Figure 3) for stability.
 * The approximate terms are evaluated in the algebraically identical
 * token-level form e^{q'.kbar_j} sum_n (1 + q'.k_{j,n} - q'.kbar_j) v_{j,n},
 * using q'.kbar_j = mean_n q'.k_{j,n}, so Q, K, V and S_i are the only inputs.
 *
 * q, k, v   [heads, n, d] of `in_dtype`, 16-byte aligned.
 * scale     softmax scale s > 0 (normally 1/sqrt(d)).
 * idx, cnt  the route (pisa_route layout); entries must be in [0, nb).
 * out       [heads, n, d] of `out_dtype`, 16-byte aligned.
 * bf16 inputs (d = 64 or 128) run on the tcgen05 tensor-core kernel; float32
 * inputs run in float32 arithmetic on the CUDA cores.
 * Errors: INVALID_ARG / UNSUPPORTED as for the other calls; a route entry
 * outside [0, nb) is reported through dev_status as PISA_ERR_DEVICE_CHECK and
 * that block list entry is ignored.
 */
int pisa_forward(const void* q, const void* k, const void* v, int in_dtype,
                 int heads, int n, int d, int block, float scale,
                 const int32_t* idx, const int32_t* cnt, int max_sel,
                 void* out, int out_dtype,
                 int32_t* dev_status, void* stream);

/*
 * pisa_route_ex - pisa_route with forced sink blocks and optional extra score
 * terms: the covariance bias and a per-pair bonus.
 *
 * Sources: the Piecewise-Taylor-Attention README ("Knobs": n_sink_blocks=n
 * forces the first n key blocks, e.g. an MMDiT text prefix, into the exact
 * branch; "Router polish": the second-order spread enters the ranking as the
 * bounded bonus min(w, ln B)); routing as pisa_route (Algorithm 1 step 2) and,
 * with mnorm, as pisa_route_covariance (Section 3.3 Eq. 11).
 *
 * S_i = band(i) U {0, ..., n_sink - 1} U top_k of the remaining blocks by
 * r_ij = s qbar_i . kbar_j [+ log(mnorm_j + eps)] [+ bonus_ij].
 * mnorm      optional [heads, nb] float32 (NULL: no covariance term); eps as
 *            pisa_route_covariance (ignored when mnorm is NULL).
 * bonus      optional [heads, nb, nb] float32, row i = query block (e.g. the
 *            wrank output of pisa_second_order_spread); NULL: none.
 * n_sink     >= 0 (values above nb mean every block).
 * max_sel    >= min(nb, topk + 2 band + 1 + n_sink).
 * Scores are screened in float32 with a bound that covers every rounding and
 * the ambiguous candidates are re-scored in double-float, as in pisa_route.
 * Other arguments, outputs and errors: as pisa_route.
 */
int pisa_route_ex(const float* qbar, const float* kbar, const float* mnorm, float eps,
                  const float* bonus, int heads, int nb, int d, float scale, int topk,
                  int band, int n_sink, int32_t* idx, int32_t* cnt, int max_sel,
                  int32_t* dev_status, void* stream);

/*
 * pisa_morton_permutation - Morton (Z-order) token order of a T x Y x X grid.
 *
 * Source: the Piecewise-Taylor-Attention README ("Morton tile reorder + fused
 * gather kernel"; the protocol's "Morton (Z-order) tile reordering").
 *
 * perm       [n_prefix + t*y*x] int32 out: perm[p] = source index of the
 *            token placed at position p. The first n_prefix tokens (a text
 *            prefix) keep their places; grid token (ti, yi, xi), source index
 *            n_prefix + (ti*y + yi)*x + xi, goes to n_prefix + its rank in the
 *            order of the code interleaving the bits of ti, yi, xi (bit b of ti
 *            at position 3b + 2, of yi at 3b + 1, of xi at 3b).
 * Errors: INVALID_ARG for a null perm or sizes < 1 (n_prefix < 0);
 * UNSUPPORTED above 2^20 tokens.
 */
int pisa_morton_permutation(int t, int y, int x, int n_prefix, int32_t* perm,
                            int32_t* dev_status, void* stream);

/*
 * pisa_reorder_heads - fused token gather and transpose into the per-head
 * layout: out[h][p][:] = x[perm[p]][h][:].
 * pisa_restore_heads - the inverse: y[perm[p]][h][:] = o[h][p][:].
 *
 * Source: the Piecewise-Taylor-Attention README ("a single kernel fuses the
 * [B,T,H,D]->[B,H,T,D] transpose with the token gather and its inverse").
 *
 * x, y       [n, heads, d] of `dtype` (token-major, the model's layout).
 * out, o     [heads, n, d] of `dtype` (the layout of the attention calls).
 * perm       [n] int32, a permutation of 0..n-1 (pisa_morton_permutation);
 *            entries outside [0, n) are skipped and reported as
 *            PISA_ERR_DEVICE_CHECK in *dev_status.
 * All buffers 16-byte aligned; d * element size must be a multiple of 16
 * bytes (UNSUPPORTED otherwise). The copy is bit-exact.
 */
int pisa_reorder_heads(const void* x, int dtype, int n, int heads, int d, const int32_t* perm,
                       void* out, int32_t* dev_status, void* stream);
int pisa_restore_heads(const void* o, int dtype, int n, int heads, int d, const int32_t* perm,
                       void* y, int32_t* dev_status, void* stream);

/*
 * pisa_second_order_spread - second-order correction of the block mass.
 *
 * Source: the Piecewise-Taylor-Attention README ("Blog post"): the mass of an
 * approximated block, n_j e^{q'.kbar_j} in Section 3.2 Eq. 3 of the PISA
 * paper, becomes n_j e^{q'.kbar_j + w_ij} with
 *   w_ij = 1/2 s^2 sum_c qsq_{i,c} kvar_{j,c},
 * qsq_i the per-channel mean of q^2 over query block i and kvar_j the
 * per-channel variance (1/n_j) of the keys of block j; w_ij is set to 0 where
 * it exceeds ln n_j (the README's gate).
 *
 * q, k      [heads, n, d] of `in_dtype`, 16-byte aligned.
 * scale     s > 0.
 * kbar      [heads, nb, d] float32 (pisa_block_stats).
 * qsq, kvar [heads, nb, d] float32 out, 16-byte aligned.
 * w         [heads, nb, nb] float32 out (row i = query block), 16-byte aligned:
 *           the gated spread for pisa_forward_second_order.
 * wrank     optional [heads, nb, nb] float32 out: min(w_ij, ln n_j), the
 *           README's ranking bonus for pisa_route_ex (NULL: not written).
 * Sums are float32; the gate is decided on the float32 w.
 * Errors: as pisa_block_stats; INVALID_ARG for scale <= 0 or not finite.
 */
int pisa_second_order_spread(const void* q, const void* k, int in_dtype,
                             int heads, int n, int d, int block, float scale,
                             const float* kbar, float* qsq, float* kvar, float* w,
                             float* wrank, int32_t* dev_status, void* stream);

/*
 * pisa_forward_second_order - pisa_forward with the second-order block mass.
 *
 * Every approximated block j of query block i enters with the logit
 * q'.kbar_j + w_ij instead of q'.kbar_j: mass n_j e^{a + w}, Taylor numerator
 * e^{a + w} (Vhat_j + q' H_j) (the README's "virtual-token logits"); exact
 * blocks are unchanged.
 *
 * w          [heads, nb, nb] float32 (pisa_second_order_spread, or any
 *            caller-chosen spread), 16-byte aligned.
 * Other arguments, layouts and errors: as pisa_forward.
 */
int pisa_forward_second_order(const void* q, const void* k, const void* v, int in_dtype,
                              int heads, int n, int d, int block, float scale,
                              const int32_t* idx, const int32_t* cnt, int max_sel,
                              const float* w, void* out, int out_dtype,
                              int32_t* dev_status, void* stream);

/*
 * pisa_forward_hybrid - the hybrid-order output (global first-order term).
 *
 * Source: Section 3.3 "Global First-Order Correction", Eq. 9-10, and
 * Algorithm 1 Phase 3: the block-wise zeroth-order terms are kept and the
 * block-wise first-order matrices are replaced by their global mean:
 *   D_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} + sum_{j not in S_i} n_j alpha_tj
 *   N_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} v_{j,n}
 *       + sum_{j not in S_i} alpha_tj Vhat_j + (sum_{j not in S_i} alpha_tj) q' Hbar
 *   o_t = N_t / D_t,   alpha_tj = e^{q'.kbar_j},   q' = s q_t.
 * Its error against pisa_forward is bounded by Theorem 3.1 (Appendix C).
 *
 * q, k, v, scale, idx, cnt, max_sel, out, out_dtype: as pisa_forward.
 * kbar, vsum [heads, nb, d] float32 (pisa_block_stats); hbar [heads, d, d]
 * float32 (pisa_global_first_order).
 * workspace  device scratch owned by the caller, 16-byte aligned, of at least
 *            pisa_forward_hybrid_workspace_size() bytes (NULL when that is 0).
 *            bf16 inputs (d = 64 or 128) run on the tcgen05 tensor-core kernel,
 *            which first writes bf16 hi + lo copies of kbar, vsum and hbar
 *            there (kbar and Vhat enter the tensor cores as two bf16 terms so
 *            the centroid logits keep ~16 significant bits), followed by the
 *            plan of the kernel's work: query blocks whose critical sets
 *            overlap most share a 128-row tile, and tiles with similar
 *            numbers of exact key tiles share a CTA (the plan decides where a
 *            row is computed, never its value). Other inputs run
 *            in float32 on the CUDA cores and need no workspace. The contents
 *            are overwritten; concurrent calls need separate workspaces.
 * Errors: as pisa_forward; INVALID_ARG for a missing or too small workspace;
 * UNSUPPORTED when the union of four query blocks' critical sets cannot be
 * staged in shared memory (more than ~12000 critical blocks).
 */
int pisa_forward_hybrid(const void* q, const void* k, const void* v, int in_dtype,
                        int heads, int n, int d, int block, float scale,
                        const float* kbar, const float* vsum, const float* hbar,
                        const int32_t* idx, const int32_t* cnt, int max_sel,
                        void* out, int out_dtype,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, void* stream);

/* Bytes of workspace pisa_forward_hybrid needs for these arguments (0 if none). */
size_t pisa_forward_hybrid_workspace_size(int in_dtype, int heads, int n, int d);

/*
 * pisa_forward_hybrid_static - pisa_forward_hybrid for callers that cannot
 * allocate device memory.
 *
 * The paper has no counterpart to this call: it is a packaging variant of
 * pisa_forward_hybrid. That call needs a scratch buffer which the caller must
 * allocate. Code that is handed only its input and output pointers and may
 * not allocate device memory itself (a plugin inside a framework that owns
 * every device allocation, a process whose allocator belongs to another
 * runtime, a component that must not change the device footprint at run
 * time) can call this variant instead: same inputs, outputs and result, no
 * workspace argument, and no allocation of any kind. Its scratch is a
 * file-scope device array of pisa_forward_hybrid_static_capacity() bytes
 * (48 MiB) for the bf16 operand copies, plus a 384 KiB one for the plan of
 * query tiles (always large enough when the operands fit), that every GPU
 * loading the library holds until the process exits.
 *
 * - All calls share that array and every call overwrites it: calls whose
 *   kernels could overlap on the GPU (other streams, other host threads) race
 *   and must be serialised by the caller. Nothing has to be cleared between
 *   calls (each call writes all the scratch it reads).
 * - Every call looks up the array's device address (no allocation) on the
 *   device current at the call. The first call on a device also loads the
 *   library's device code there; make that first call before any stream
 *   capture.
 * - Inputs whose pisa_forward_hybrid_workspace_size() is 0 need no scratch
 *   and run exactly as in pisa_forward_hybrid.
 * Errors: as pisa_forward_hybrid; UNSUPPORTED (with a pisa_last_error()
 * message) when the operand copies these sizes need exceed the array.
 */
int pisa_forward_hybrid_static(const void* q, const void* k, const void* v, int in_dtype,
                               int heads, int n, int d, int block, float scale,
                               const float* kbar, const float* vsum, const float* hbar,
                               const int32_t* idx, const int32_t* cnt, int max_sel,
                               void* out, int out_dtype,
                               int32_t* dev_status, void* stream);

/* Size in bytes of the fixed operand scratch array of pisa_forward_hybrid_static. */
size_t pisa_forward_hybrid_static_capacity(void);

/*
 * pisa_attention_host - statistics, route and block-wise forward (pisa_block_stats,
 * pisa_route, pisa_forward in that order) on Q, K, V in HOST memory, with
 * the output written to HOST memory: the path as one call for code that
 * keeps its tensors on the host.
 *
 * Source: the three calls' passages (Section 3.2 Eq. (3)-(6); Figure 4
 * "Prepare Phase", Algorithm 1 step 2); the band as in pisa_route.
 *
 * q, k, v    HOST [heads, n, d] of `in_dtype`; out HOST [heads, n, d] of
 *            `out_dtype`. Page-locked (pinned) memory lets the copies overlap
 *            the compute; pageable memory works but its copies do not overlap.
 *            The buffers must stay valid until `stream` has passed this call.
 * scale, topk, band: as pisa_route / pisa_forward.
 * groups     1..64: heads go through in that many contiguous groups; group
 *            c + 1 is uploaded and group c - 1 downloaded while group c is
 *            computed. taper != 0 gives the first and the last group half the
 *            weight of the others (their copies are the ones nothing hides).
 * workspace  DEVICE scratch owned by the caller, 256-byte aligned, of at least
 *            pisa_attention_host_workspace_size() bytes: two groups' inputs,
 *            statistics, route and output. Calls that overlap on the GPU need
 *            separate workspaces.
 * The call enqueues copies and kernels on streams and events of its own,
 * created for the call and released once their work is done; `stream` (the
 * caller's) waits for all of it, and everything already on `stream` runs
 * first. The result is the same as the three device calls on the whole
 * tensors, bit for bit (heads are independent). Errors: INVALID_ARG /
 * UNSUPPORTED as the three calls, INVALID_ARG for a missing, misaligned or
 * short workspace or groups outside 1..64 (with a pisa_last_error()
 * message); on an error after work was enqueued, that work may still run:
 * synchronise before reusing the buffers.
 */
int pisa_attention_host(const void* q, const void* k, const void* v, int in_dtype,
                        int heads, int n, int d, int block, float scale, int topk, int band,
                        void* out, int out_dtype, int groups, int taper,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, void* stream);

/* Bytes of workspace pisa_attention_host needs for these arguments (0 for
 * invalid sizes). */
size_t pisa_attention_host_workspace_size(int in_dtype, int out_dtype, int heads, int n, int d,
                                          int topk, int band, int groups, int taper);

/* Static, human-readable name of a pisa_status code. */
const char* pisa_status_string(int status);

/* Description of the last PISA_ERR_CUDA returned to the calling host thread
 * (the failing CUDA call, its error code and message), or of the last scratch
 * size rejected by pisa_forward_hybrid_static; "no error" before any. The
 * string is owned by the library and stays valid until the thread's next
 * failing call. */
const char* pisa_last_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int pisa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PISA_H */
