// Internal launcher declarations (host side). Arguments are validated by the
// C ABI layer (api.cu) before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pisa {

int launch_block_stats(const void* q, const void* k, const void* v, int in_bf16, int heads,
                       int n, int d, float* qbar, float* kbar, float* vsum, void* hmat,
                       int h_bf16, int32_t* status, cudaStream_t stream);

// mnorm (optional, [heads, nb]): rank by s qbar.kbar + log(mnorm + eps)
// instead of qbar.kbar.
int launch_route(const float* qbar, const float* kbar, int heads, int nb, int d, int topk,
                 int band, int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
                 cudaStream_t stream, const float* mnorm = nullptr, float eps = 0.f,
                 float scale = 1.f, int n_sink = 0, const float* bonus = nullptr);

// Morton position of every grid token (perm[p] = source index), prefix kept.
int launch_morton_permutation(int T, int Y, int X, int n_prefix, int32_t* perm,
                              cudaStream_t stream);
// gather: dst[h][p] = src[perm[p]][h]; scatter: dst[perm[p]][h] = src[h][p];
// rows of row_bytes (a multiple of 16).
int launch_heads_copy(const void* src, void* dst, int gather, int n, int heads, int row_bytes,
                      const int32_t* perm, int32_t* dev_status, cudaStream_t stream);

// M_j = ||H_j - Hbar|| per (head, block) into mnorm [heads, nb]; spectral or
// Frobenius norm.
// H_j of bf16 inputs with d = 128 on the tensor cores, from the block means
// kbar (launch_block_stats runs the means first).
int launch_block_h_tc(const void* k, const void* v, int heads, int n, const float* kbar,
                      void* hmat, int h_bf16, int32_t* status, cudaStream_t stream);
int launch_block_heterogeneity(const void* k, const void* v, int in_bf16, int heads, int n,
                               int d, const float* kbar, const float* hbar, int spectral,
                               float* mnorm, int32_t* status, cudaStream_t stream);

// float32 CUDA-core forward (float32 inputs; any supported d).
int launch_forward_simt(const void* q, const void* k, const void* v, int heads,
                        int n, int d, float scale, const int32_t* idx, const int32_t* cnt,
                        int max_sel, void* out, int out_bf16, int32_t* dev_status,
                        cudaStream_t stream, const float* spread = nullptr);

// tcgen05 / TMEM / TMA forward for bf16 inputs, d = 64 or 128. `spread` (optional,
// [heads, nb, nb]): second-order logit shift of the approximated blocks.
int launch_forward_tc(const void* q, const void* k, const void* v, int heads, int n, int d,
                      float scale, const int32_t* idx, const int32_t* cnt, int max_sel,
                      void* out, int out_bf16, int32_t* dev_status, cudaStream_t stream,
                      const float* spread = nullptr);

// Second-order statistics: qsq / kvar [heads, nb, d] (mean of q^2 per query
// block, key variance per key block) and the gated spread w [heads, nb, nb].
int launch_second_order(const void* q, const void* k, int in_bf16, int heads, int n, int d,
                        float scale, const float* kbar, float* qsq, float* kvar, float* w,
                        float* wrank, cudaStream_t stream);

// hybrid-order forward (global Hbar), float32 CUDA cores.
int launch_forward_hybrid_simt(const void* q, const void* k, const void* v,
                               int heads, int n, int d, float scale, const float* kbar,
                               const float* vsum, const float* hbar, const int32_t* idx,
                               const int32_t* cnt, int max_sel, void* out, int out_bf16,
                               int32_t* dev_status, cudaStream_t stream);

// hybrid-order forward on tcgen05 (bf16, d = 64 or 128). `workspace` takes
// forward_hybrid_tc_operand_bytes() (the bf16 hi/lo operand copies, 16-byte
// aligned) and `plan` forward_hybrid_tc_plan_bytes() (the query blocks of
// every CTA, 4-byte aligned); forward_hybrid_tc_workspace() is the size
// of one buffer holding both, the plan at the first 256-byte boundary after
// the operands.
size_t forward_hybrid_tc_operand_bytes(int heads, int n, int d);
// The plan of that kernel for nb query blocks per head (hybrid_plan.cu):
// plan [heads][ceil(n / 256)][4] query block indices, nb = none; at most
// kHybridPlanMaxTiles 128-row query tiles per head (n <= 2^20).
constexpr int kHybridPlanMaxTiles = 8192;
int launch_hybrid_plan(const int32_t* idx, const int32_t* cnt, int heads, int nb, int max_sel,
                       int32_t* plan, cudaStream_t stream);
size_t forward_hybrid_tc_plan_bytes(int heads, int n);
size_t forward_hybrid_tc_workspace(int heads, int n, int d);
int launch_forward_hybrid_tc(const void* q, const void* k, const void* v, int heads, int n, int d,
                             float scale, const float* kbar, const float* vsum, const float* hbar,
                             const int32_t* idx, const int32_t* cnt, int max_sel, void* out,
                             int out_bf16, void* workspace, int32_t* plan, int32_t* dev_status,
                             cudaStream_t stream);

// The same with the scratch in a fixed file-scope device array (no allocation).
int forward_hybrid_static(const void* q, const void* k, const void* v, int heads, int n, int d,
                          float scale, const float* kbar, const float* vsum, const float* hbar,
                          const int32_t* idx, const int32_t* cnt, int max_sel, void* out,
                          int out_bf16, int32_t* dev_status, cudaStream_t stream);
size_t forward_hybrid_static_capacity();

// Hbar = (1/nb) sum_j H_j per head into hbar [heads, d, d]; every element is
// written once by a cluster-wide reduction, so hbar needs no zeroing.
int launch_global_h(const void* k, const void* v, int in_bf16, int heads, int n, int d,
                    const float* kbar, const float* vsum, float* hbar, int32_t* dev_status,
                    cudaStream_t stream);

}  // namespace pisa
