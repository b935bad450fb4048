// Token reorder of the Piecewise-Taylor-Attention README ("Morton tile
// reorder + fused gather kernel"): grid tokens in Morton (Z) order so that a
// 64-token block covers a compact 3-D neighbourhood, fused with the transpose
// between the model's token-major [N, H, d] layout and the per-head [H, N, d]
// layout the attention kernels read.
//
// morton_rank_kernel: the Morton position of every grid token computed
//   directly, without sorting: walking the octant digits of the token's code
//   from the top (digit = 4 t_b + 2 y_b + x_b, t the most significant), the
//   rank grows at each level by the number of grid points in the sibling
//   octants with a smaller digit; a cube cell holds the product over the
//   three axes of its overlap with [0, T), [0, Y), [0, X). O(8 log2 side) per
//   token, exact, no scratch memory.
// gather_heads_kernel / scatter_heads_kernel: one warp per token, 16-byte
//   vectors; the gather reads the token's contiguous H x d row and writes one
//   d-row per head, the scatter the reverse.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

__device__ __forceinline__ long long overlap(long long a, long long s, long long len) {
  return a >= len ? 0 : (a + s < len ? s : len - a);
}

__global__ void morton_rank_kernel(int T, int Y, int X, int bits, int n_prefix,
                                   int32_t* __restrict__ perm) {
  const long long total = static_cast<long long>(T) * Y * X;
  for (long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; r < total;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(r / (static_cast<long long>(Y) * X));
    const int y = static_cast<int>((r / X) % Y);
    const int x = static_cast<int>(r % X);
    long long rank = 0;
    long long t0 = 0, y0 = 0, x0 = 0;  // corner of the current cell
    for (int b = bits - 1; b >= 0; --b) {
      const long long s = 1ll << b;  // side of the child cells
      const int dt = (t >> b) & 1, dy = (y >> b) & 1, dx = (x >> b) & 1;
      const int digit = 4 * dt + 2 * dy + dx;
      for (int o = 0; o < digit; ++o) {
        const long long ct = overlap(t0 + ((o >> 2) & 1) * s, s, T);
        const long long cy = overlap(y0 + ((o >> 1) & 1) * s, s, Y);
        const long long cx = overlap(x0 + (o & 1) * s, s, X);
        rank += ct * cy * cx;
      }
      t0 += dt * s;
      y0 += dy * s;
      x0 += dx * s;
    }
    perm[n_prefix + rank] = static_cast<int32_t>(n_prefix + r);
  }
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_prefix; p += gridDim.x * blockDim.x)
    perm[p] = p;
}

constexpr int kWarps = 8;

// out[h][p] = x[perm[p]][h] (gather) or y[perm[p]][h] = o[h][p] (scatter);
// rows of `row16` 16-byte vectors.
template <bool GATHER>
__global__ void __launch_bounds__(kWarps * 32)
heads_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int n, int heads, int row16,
             const int32_t* __restrict__ perm, int32_t* status) {
  const int lane = threadIdx.x % 32;
  const int per_token = heads * row16;
  for (int p = blockIdx.x * kWarps + threadIdx.x / 32; p < n; p += gridDim.x * kWarps) {
    const int tok = perm[p];
    if (tok < 0 || tok >= n) {
      if (lane == 0) report(status, PISA_ERR_DEVICE_CHECK);
      continue;
    }
    for (int e = lane; e < per_token; e += 32) {
      const int h = e / row16, c = e % row16;
      const size_t token_major = static_cast<size_t>(tok) * per_token + e;
      const size_t head_major = (static_cast<size_t>(h) * n + p) * row16 + c;
      if (GATHER)
        dst[head_major] = __ldg(src + token_major);
      else
        dst[token_major] = __ldg(src + head_major);
    }
  }
}

}  // namespace

int launch_morton_permutation(int T, int Y, int X, int n_prefix, int32_t* perm,
                              cudaStream_t stream) {
  int bits = 1;
  while ((1 << bits) < T || (1 << bits) < Y || (1 << bits) < X) ++bits;
  const long long total = static_cast<long long>(T) * Y * X + n_prefix;
  const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 152 * 16));
  morton_rank_kernel<<<blocks, 256, 0, stream>>>(T, Y, X, bits, n_prefix, perm);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

int launch_heads_copy(const void* src, void* dst, int gather, int n, int heads, int row_bytes,
                      const int32_t* perm, int32_t* dev_status, cudaStream_t stream) {
  const int row16 = row_bytes / 16;
  const int blocks = std::max(1, std::min((n + kWarps - 1) / kWarps, 152 * 16));
  if (gather)
    heads_kernel<true><<<blocks, kWarps * 32, 0, stream>>>(static_cast<const uint4*>(src),
                                                           static_cast<uint4*>(dst), n, heads,
                                                           row16, perm, dev_status);
  else
    heads_kernel<false><<<blocks, kWarps * 32, 0, stream>>>(static_cast<const uint4*>(src),
                                                            static_cast<uint4*>(dst), n, heads,
                                                            row16, perm, dev_status);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace pisa
