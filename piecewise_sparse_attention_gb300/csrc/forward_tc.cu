// bf16 d=128 forward. Until the tensor-core kernel lands, this entry runs the
// float32 CUDA-core kernel.
#include "common.cuh"
#include "kernels.h"

namespace pisa {

int launch_forward_tc(const void* q, const void* k, const void* v, int heads, int n, int d,
                      float scale, const int32_t* idx, const int32_t* cnt, int max_sel,
                      void* out, int out_bf16, int32_t* dev_status, cudaStream_t stream) {
  return launch_forward_simt(q, k, v, 1, heads, n, d, scale, idx, cnt, max_sel, out, out_bf16,
                             dev_status, stream);
}

}  // namespace pisa
