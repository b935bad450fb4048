// pisa_forward_hybrid_static: the hybrid-order forward for callers that cannot
// allocate device memory.
//
// pisa_forward_hybrid needs a scratch buffer (the bf16 hi/lo copies of kbar,
// Vhat and Hbar that its tensor-core kernel reads through TMA, and the pairing
// of query tiles into CTAs) and expects the caller to provide it. Some callers have no way to do that: code that runs
// where device allocation is not allowed or not available (a plugin handed
// only its input and output pointers by a host framework that owns all device
// memory, a process whose allocator is reserved for another runtime, code that
// must not grow the device footprint at run time). This entry point takes the
// same inputs and outputs but keeps its scratch in one file-scope __device__
// array of fixed size for the operand copies and one for the pairing, so it
// never allocates: no cudaMalloc / cudaFree and no allocating library call.
//
// Consequences for the caller:
// * every GPU that loads this library holds the arrays (kStaticScratchBytes
//   and kStaticPlanBytes) until the process exits;
// * the arrays are shared by all calls: two calls whose kernels overlap on the
//   GPU (different streams, or different host threads) race on it and must be
//   serialised by the caller. Every byte the kernel reads is written earlier
//   in the same call, so nothing needs clearing between calls;
// * every call looks up the array's device address (cudaGetSymbolAddress,
//   which allocates nothing) on the device current at the call, so the
//   address stays right after a context reset; the first call on a device
//   also loads the library's device code there, so make that first call
//   before any stream capture.
#include "common.cuh"
#include "kernels.h"

namespace pisa {

// 48 MiB covers every workload shipped with this library (the largest, 16
// heads x 131072 tokens, needs 34.6 MB).
constexpr size_t kStaticScratchBytes = size_t(48) << 20;
// The pairing takes 16 bytes per 256 query rows (rounded up) and head; the
// operand copies take at least 512 bytes per 64 rows and 32 KiB per head, so
// the pairing is at most 1/128 of them and 384 KiB covers every size whose
// operands fit the scratch array.
constexpr size_t kStaticPlanBytes = kStaticScratchBytes / 128;

namespace {

__device__ __align__(256) unsigned char g_hybrid_scratch[kStaticScratchBytes];
__device__ __align__(256) int32_t g_hybrid_plan[kStaticPlanBytes / sizeof(int32_t)];

// Device addresses of the arrays in the current device's context. In host
// code the symbols are only host-side stand-ins; the kernel must be given
// these addresses. Looked up on every call: a cached address would dangle
// after cudaDeviceReset re-creates the context and reloads the module.
int scratch_address(void** scratch, int32_t** plan) {
  void* p = nullptr;
  PISA_CUDA_TRY(cudaGetSymbolAddress(&p, g_hybrid_scratch));
  *scratch = p;
  PISA_CUDA_TRY(cudaGetSymbolAddress(&p, g_hybrid_plan));
  *plan = static_cast<int32_t*>(p);
  return PISA_OK;
}

}  // namespace

int forward_hybrid_static(const void* q, const void* k, const void* v, int heads, int n, int d,
                          float scale, const float* kbar, const float* vsum, const float* hbar,
                          const int32_t* idx, const int32_t* cnt, int max_sel, void* out,
                          int out_bf16, int32_t* dev_status, cudaStream_t stream) {
  const size_t need = forward_hybrid_tc_operand_bytes(heads, n, d);
  if (need > kStaticScratchBytes) {
    note_error("pisa_forward_hybrid_static: needs %zu bytes of scratch, above its fixed %zu",
               need, kStaticScratchBytes);
    return PISA_ERR_UNSUPPORTED;
  }
  if (forward_hybrid_tc_plan_bytes(heads, n) > kStaticPlanBytes) {  // implied by the check above
    note_error("pisa_forward_hybrid_static: needs %zu bytes of scratch for the tile pairing, "
               "above its fixed %zu", forward_hybrid_tc_plan_bytes(heads, n), kStaticPlanBytes);
    return PISA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  int32_t* plan = nullptr;
  const int rc = scratch_address(&scratch, &plan);
  if (rc != PISA_OK) return rc;
  return launch_forward_hybrid_tc(q, k, v, heads, n, d, scale, kbar, vsum, hbar, idx, cnt,
                                  max_sel, out, out_bf16, scratch, plan, dev_status, stream);
}

size_t forward_hybrid_static_capacity() { return kStaticScratchBytes; }

}  // namespace pisa
