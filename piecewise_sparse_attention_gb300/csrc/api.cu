// C ABI of the library (declared in include/pisa.h): argument validation on
// the host, then one or two kernel launches on the caller's stream. Nothing
// here allocates device memory or synchronises.
#include <math.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pisa.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kMaxHeads = 65535;     // grid.y limit of the per-head launches
constexpr int kMaxTokens = 1 << 20;  // 16384 blocks of 64 tokens
constexpr int kMaxBlocks = kMaxTokens / pisa::kBlock;

thread_local char g_last_error[256] = "no error";

// An NVTX range named after the entry point around each call that enqueues
// work, so that a timeline tool shows the host-side call above its kernels.
// Without a tool attached a push or pop is a call through an empty hook.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(int dt) { return dt == PISA_F32 || dt == PISA_BF16; }

int check_shape(int heads, int n, int d, int block) {
  if (heads < 1 || heads > kMaxHeads || n < 1 || block != pisa::kBlock) return PISA_ERR_INVALID_ARG;
  if (n > kMaxTokens) return PISA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  return PISA_OK;
}

bool in_aligned(const void* q, const void* k, const void* v) {
  return q && k && v && aligned16(q) && aligned16(k) && aligned16(v);
}

}  // namespace

namespace pisa {
int cuda_fail(const char* what, int code, const char* detail) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: error %d (%s)", what, code,
           detail ? detail : "");
  return PISA_ERR_CUDA;
}

void note_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}
}  // namespace pisa

extern "C" {

int pisa_version(void) { return 100; }

const char* pisa_last_error(void) { return g_last_error; }

const char* pisa_status_string(int status) {
  switch (status) {
    case PISA_OK: return "ok";
    case PISA_ERR_INVALID_ARG: return "invalid argument";
    case PISA_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PISA_ERR_CUDA: return "CUDA error";
    case PISA_ERR_TIMEOUT: return "device wait timed out";
    case PISA_ERR_DEVICE_CHECK: return "device bounds check failed";
    default: return "unknown status";
  }
}

int pisa_block_stats(const void* q, const void* k, const void* v, int in_dtype, int heads, int n,
                     int d, int block, float* qbar, float* kbar, float* vsum, void* hmat,
                     int h_dtype, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_block_stats");
  if (!dtype_ok(in_dtype)) return PISA_ERR_INVALID_ARG;
  if (!in_aligned(q, k, v)) return PISA_ERR_INVALID_ARG;
  if (!qbar && !kbar && !vsum && !hmat) return PISA_ERR_INVALID_ARG;
  if ((qbar && !aligned16(qbar)) || (kbar && !aligned16(kbar)) || (vsum && !aligned16(vsum)) ||
      (hmat && !aligned16(hmat)))
    return PISA_ERR_INVALID_ARG;
  if (hmat && !dtype_ok(h_dtype)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  return pisa::launch_block_stats(q, k, v, in_dtype == PISA_BF16, heads, n, d, qbar, kbar, vsum,
                                  hmat, h_dtype == PISA_BF16, dev_status,
                                  static_cast<cudaStream_t>(stream));
}

int pisa_global_first_order(const void* k, const void* v, int in_dtype, int heads, int n, int d,
                            int block, const float* kbar, const float* vsum, float* hbar,
                            int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_global_first_order");
  if (!dtype_ok(in_dtype)) return PISA_ERR_INVALID_ARG;
  if (!k || !v || !aligned16(k) || !aligned16(v) || !kbar || !vsum || !hbar ||
      !aligned16(kbar) || !aligned16(vsum) || !aligned16(hbar))
    return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  return pisa::launch_global_h(k, v, in_dtype == PISA_BF16, heads, n, d, kbar, vsum, hbar,
                               dev_status, static_cast<cudaStream_t>(stream));
}

int pisa_route(const float* qbar, const float* kbar, int heads, int nb, int d, float scale,
               int topk, int band, int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
               void* stream) {
  NvtxRange nvtx_range("pisa_route");
  if (!qbar || !kbar || !idx || !cnt || !aligned16(qbar) || !aligned16(kbar))
    return PISA_ERR_INVALID_ARG;
  if (heads < 1 || heads > kMaxHeads || nb < 1 || topk < 0 || band < 0) return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  if (nb > kMaxBlocks) return PISA_ERR_UNSUPPORTED;
  const long long need = static_cast<long long>(topk) + 2LL * band + 1LL;
  const long long min_sel = need < nb ? need : nb;
  if (max_sel < min_sel) return PISA_ERR_INVALID_ARG;
  return pisa::launch_route(qbar, kbar, heads, nb, d, topk, band, idx, cnt, max_sel, dev_status,
                            static_cast<cudaStream_t>(stream));
}

int pisa_block_heterogeneity(const void* k, const void* v, int in_dtype, int heads, int n, int d,
                             int block, const float* kbar, const float* hbar, int norm,
                             float* mnorm, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_block_heterogeneity");
  if (!dtype_ok(in_dtype)) return PISA_ERR_INVALID_ARG;
  if (norm != PISA_NORM_SPECTRAL && norm != PISA_NORM_FROBENIUS) return PISA_ERR_INVALID_ARG;
  if (!k || !v || !aligned16(k) || !aligned16(v) || !kbar || !hbar || !mnorm ||
      !aligned16(kbar) || !aligned16(hbar) || !aligned16(mnorm))
    return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  return pisa::launch_block_heterogeneity(k, v, in_dtype == PISA_BF16, heads, n, d, kbar, hbar,
                                          norm == PISA_NORM_SPECTRAL, mnorm, dev_status,
                                          static_cast<cudaStream_t>(stream));
}

int pisa_route_covariance(const float* qbar, const float* kbar, const float* mnorm, float eps,
                          int heads, int nb, int d, float scale, int topk, int band,
                          int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
                          void* stream) {
  NvtxRange nvtx_range("pisa_route_covariance");
  if (!mnorm || !aligned16(mnorm)) return PISA_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !isfinite(eps)) return PISA_ERR_INVALID_ARG;
  if (!qbar || !kbar || !idx || !cnt || !aligned16(qbar) || !aligned16(kbar))
    return PISA_ERR_INVALID_ARG;
  if (heads < 1 || heads > kMaxHeads || nb < 1 || topk < 0 || band < 0) return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  if (nb > kMaxBlocks) return PISA_ERR_UNSUPPORTED;
  const long long need = static_cast<long long>(topk) + 2LL * band + 1LL;
  const long long min_sel = need < nb ? need : nb;
  if (max_sel < min_sel) return PISA_ERR_INVALID_ARG;
  return pisa::launch_route(qbar, kbar, heads, nb, d, topk, band, idx, cnt, max_sel, dev_status,
                            static_cast<cudaStream_t>(stream), mnorm, eps, scale);
}

int pisa_second_order_spread(const void* q, const void* k, int in_dtype, int heads, int n, int d,
                             int block, float scale, const float* kbar, float* qsq, float* kvar,
                             float* w, float* wrank, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_second_order_spread");
  (void)dev_status;
  if (!dtype_ok(in_dtype)) return PISA_ERR_INVALID_ARG;
  if (!q || !k || !aligned16(q) || !aligned16(k) || !kbar || !qsq || !kvar || !w ||
      !aligned16(kbar) || !aligned16(qsq) || !aligned16(kvar) || !aligned16(w) ||
      (wrank && !aligned16(wrank)))
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  return pisa::launch_second_order(q, k, in_dtype == PISA_BF16, heads, n, d, scale, kbar, qsq,
                                   kvar, w, wrank, static_cast<cudaStream_t>(stream));
}

int pisa_forward_second_order(const void* q, const void* k, const void* v, int in_dtype,
                              int heads, int n, int d, int block, float scale,
                              const int32_t* idx, const int32_t* cnt, int max_sel,
                              const float* w, void* out, int out_dtype, int32_t* dev_status,
                              void* stream) {
  NvtxRange nvtx_range("pisa_forward_second_order");
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return PISA_ERR_INVALID_ARG;
  if (!in_aligned(q, k, v) || !out || !aligned16(out) || !idx || !cnt || max_sel < 1 || !w ||
      !aligned16(w))
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in_dtype == PISA_BF16)  // d = 64 or 128: tensor cores
    return pisa::launch_forward_tc(q, k, v, heads, n, d, scale, idx, cnt, max_sel, out,
                                   out_dtype == PISA_BF16, dev_status, s, w);
  return pisa::launch_forward_simt(q, k, v, heads, n, d, scale, idx, cnt,
                                   max_sel, out, out_dtype == PISA_BF16, dev_status, s, w);
}

int pisa_route_ex(const float* qbar, const float* kbar, const float* mnorm, float eps,
                  const float* bonus, int heads, int nb, int d, float scale, int topk, int band,
                  int n_sink, int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
                  void* stream) {
  NvtxRange nvtx_range("pisa_route_ex");
  if (mnorm && (!aligned16(mnorm) || !(eps > 0.f) || !isfinite(eps))) return PISA_ERR_INVALID_ARG;
  if (bonus && !aligned16(bonus)) return PISA_ERR_INVALID_ARG;
  if (!qbar || !kbar || !idx || !cnt || !aligned16(qbar) || !aligned16(kbar))
    return PISA_ERR_INVALID_ARG;
  if (heads < 1 || heads > kMaxHeads || nb < 1 || topk < 0 || band < 0 || n_sink < 0)
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  if (nb > kMaxBlocks) return PISA_ERR_UNSUPPORTED;
  const long long need = static_cast<long long>(topk) + 2LL * band + 1LL + n_sink;
  const long long min_sel = need < nb ? need : nb;
  if (max_sel < min_sel) return PISA_ERR_INVALID_ARG;
  return pisa::launch_route(qbar, kbar, heads, nb, d, topk, band, idx, cnt, max_sel, dev_status,
                            static_cast<cudaStream_t>(stream), mnorm, eps, scale, n_sink, bonus);
}

int pisa_morton_permutation(int t, int y, int x, int n_prefix, int32_t* perm,
                            int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_morton_permutation");
  (void)dev_status;
  if (!perm || t < 1 || y < 1 || x < 1 || n_prefix < 0) return PISA_ERR_INVALID_ARG;
  const long long total = static_cast<long long>(t) * y * x + n_prefix;
  if (total > kMaxTokens) return PISA_ERR_UNSUPPORTED;
  return pisa::launch_morton_permutation(t, y, x, n_prefix, perm, static_cast<cudaStream_t>(stream));
}

static int heads_copy(const void* src, int dtype, int n, int heads, int d, const int32_t* perm,
                      void* dst, int gather, int32_t* dev_status, void* stream) {
  if (!dtype_ok(dtype) || !src || !dst || !perm || !aligned16(src) || !aligned16(dst))
    return PISA_ERR_INVALID_ARG;
  if (n < 1 || heads < 1 || d < 1) return PISA_ERR_INVALID_ARG;
  if (n > kMaxTokens || heads > kMaxHeads) return PISA_ERR_UNSUPPORTED;
  const int row_bytes = d * (dtype == PISA_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return PISA_ERR_UNSUPPORTED;
  return pisa::launch_heads_copy(src, dst, gather, n, heads, row_bytes, perm, dev_status,
                                 static_cast<cudaStream_t>(stream));
}

int pisa_reorder_heads(const void* x, int dtype, int n, int heads, int d, const int32_t* perm,
                       void* out, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_reorder_heads");
  return heads_copy(x, dtype, n, heads, d, perm, out, 1, dev_status, stream);
}

int pisa_restore_heads(const void* o, int dtype, int n, int heads, int d, const int32_t* perm,
                       void* y, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_restore_heads");
  return heads_copy(o, dtype, n, heads, d, perm, y, 0, dev_status, stream);
}

int pisa_forward(const void* q, const void* k, const void* v, int in_dtype, int heads, int n,
                 int d, int block, float scale, const int32_t* idx, const int32_t* cnt,
                 int max_sel, void* out, int out_dtype, int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_forward");
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return PISA_ERR_INVALID_ARG;
  if (!in_aligned(q, k, v) || !out || !aligned16(out) || !idx || !cnt || max_sel < 1)
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in_dtype == PISA_BF16)  // d = 64 or 128: tensor cores
    return pisa::launch_forward_tc(q, k, v, heads, n, d, scale, idx, cnt, max_sel, out,
                                   out_dtype == PISA_BF16, dev_status, s);
  return pisa::launch_forward_simt(q, k, v, heads, n, d, scale, idx, cnt,
                                   max_sel, out, out_dtype == PISA_BF16, dev_status, s);
}

size_t pisa_forward_hybrid_workspace_size(int in_dtype, int heads, int n, int d) {
  if (in_dtype != PISA_BF16 || (d != 64 && d != 128) || heads < 1 || n < 1) return 0;
  return pisa::forward_hybrid_tc_workspace(heads, n, d);
}

int pisa_forward_hybrid(const void* q, const void* k, const void* v, int in_dtype, int heads,
                        int n, int d, int block, float scale, const float* kbar,
                        const float* vsum, const float* hbar, const int32_t* idx,
                        const int32_t* cnt, int max_sel, void* out, int out_dtype,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream) {
  NvtxRange nvtx_range("pisa_forward_hybrid");
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return PISA_ERR_INVALID_ARG;
  if (!in_aligned(q, k, v) || !out || !aligned16(out) || !idx || !cnt || max_sel < 1)
    return PISA_ERR_INVALID_ARG;
  if (!kbar || !vsum || !hbar || !aligned16(kbar) || !aligned16(vsum) || !aligned16(hbar))
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t need = pisa_forward_hybrid_workspace_size(in_dtype, heads, n, d);
  if (need > 0) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PISA_ERR_INVALID_ARG;
    const size_t plan_off =
        (pisa::forward_hybrid_tc_operand_bytes(heads, n, d) + 255) & ~static_cast<size_t>(255);
    int32_t* plan = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + plan_off);
    return pisa::launch_forward_hybrid_tc(q, k, v, heads, n, d, scale, kbar, vsum, hbar, idx, cnt,
                                          max_sel, out, out_dtype == PISA_BF16, workspace, plan,
                                          dev_status, s);
  }
  return pisa::launch_forward_hybrid_simt(q, k, v, heads, n, d, scale,
                                          kbar, vsum, hbar, idx, cnt, max_sel, out,
                                          out_dtype == PISA_BF16, dev_status, s);
}

size_t pisa_forward_hybrid_static_capacity(void) { return pisa::forward_hybrid_static_capacity(); }

int pisa_forward_hybrid_static(const void* q, const void* k, const void* v, int in_dtype,
                               int heads, int n, int d, int block, float scale, const float* kbar,
                               const float* vsum, const float* hbar, const int32_t* idx,
                               const int32_t* cnt, int max_sel, void* out, int out_dtype,
                               int32_t* dev_status, void* stream) {
  NvtxRange nvtx_range("pisa_forward_hybrid_static");
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return PISA_ERR_INVALID_ARG;
  if (!in_aligned(q, k, v) || !out || !aligned16(out) || !idx || !cnt || max_sel < 1)
    return PISA_ERR_INVALID_ARG;
  if (!kbar || !vsum || !hbar || !aligned16(kbar) || !aligned16(vsum) || !aligned16(hbar))
    return PISA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PISA_ERR_INVALID_ARG;
  const int st = check_shape(heads, n, d, block);
  if (st != PISA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pisa_forward_hybrid_workspace_size(in_dtype, heads, n, d) == 0)  // no scratch needed
    return pisa::launch_forward_hybrid_simt(q, k, v, heads, n, d, scale,
                                            kbar, vsum, hbar, idx, cnt, max_sel, out,
                                            out_dtype == PISA_BF16, dev_status, s);
  return pisa::forward_hybrid_static(q, k, v, heads, n, d, scale, kbar, vsum, hbar, idx, cnt,
                                     max_sel, out, out_dtype == PISA_BF16, dev_status, s);
}

}  // extern "C"
