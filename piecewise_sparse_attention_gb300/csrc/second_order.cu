// Second-order block mass of the Piecewise-Taylor-Attention README ("Blog
// post"): for query block i and key block j,
//   w_ij = 1/2 s^2 sum_c qsq_{i,c} kvar_{j,c},
//   qsq_i  = mean over the queries of block i of q^2 (per channel),
//   kvar_j = variance of the keys of block j (per channel, over its n_j tokens),
// gated to 0 where w_ij > ln n_j (the README's gate; below it the block's mass
// is n_j e^{a + w}, above it the zeroth-order n_j e^{a}); optionally also the
// route's bounded bonus min(w_ij, ln n_j). On top of "PISA:
// Piecewise Sparse Attention Is Wiser for Efficient Diffusion Transformers",
// Section 3.2 Eq. 3-6, whose block mass is n_j e^{a}.
//
// sq_var_kernel: one CTA per (block, head), one thread per channel, float32
//   sums of the block's 64 rows (coalesced row reads);
// spread_kernel: 32 x 32 tiles of w per CTA, float32 dot products over d with
//   four partial sums, then the gate.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

template <typename T>
__device__ __forceinline__ float ld(const T* p) {
  if constexpr (sizeof(T) == 2)
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
  else
    return *reinterpret_cast<const float*>(p);
}

template <typename T, int D>
__global__ void __launch_bounds__(D)
sq_var_kernel(const T* __restrict__ q, const T* __restrict__ k, const float* __restrict__ kbar,
              int n, int nb, float* __restrict__ qsq, float* __restrict__ kvar) {
  const int j = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int r0 = j * kBlock, nj = min(kBlock, n - r0);
  const size_t base = (static_cast<size_t>(h) * n + r0) * D + c;
  const float kb = kbar[(static_cast<size_t>(h) * nb + j) * D + c];
  float qs[4] = {0.f, 0.f, 0.f, 0.f}, ks[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int r = 0; r < nj; ++r) {
    const float x = ld(q + base + static_cast<size_t>(r) * D);
    const float y = ld(k + base + static_cast<size_t>(r) * D) - kb;
    qs[r & 3] = fmaf(x, x, qs[r & 3]);
    ks[r & 3] = fmaf(y, y, ks[r & 3]);
  }
  const float inv = 1.f / static_cast<float>(nj);
  const size_t o = (static_cast<size_t>(h) * nb + j) * D + c;
  qsq[o] = ((qs[0] + qs[1]) + (qs[2] + qs[3])) * inv;
  kvar[o] = ((ks[0] + ks[1]) + (ks[2] + ks[3])) * inv;
}

constexpr int kTile = 32;

template <int D>
__global__ void __launch_bounds__(256)
spread_kernel(const float* __restrict__ qsq, const float* __restrict__ kvar, int n, int nb,
              float half_s2, float* __restrict__ w, float* __restrict__ wrank) {
  __shared__ float sq[kTile][D];
  __shared__ float sk[kTile][D + 1];
  const int h = blockIdx.z, i0 = blockIdx.y * kTile, j0 = blockIdx.x * kTile;
  const int tid = threadIdx.x, ty = tid / 32, tx = tid % 32;
  for (int e = tid; e < kTile * D; e += 256) {
    const int r = e / D, c = e % D;
    sq[r][c] = (i0 + r < nb) ? qsq[(static_cast<size_t>(h) * nb + i0 + r) * D + c] : 0.f;
    sk[r][c] = (j0 + r < nb) ? kvar[(static_cast<size_t>(h) * nb + j0 + r) * D + c] : 0.f;
  }
  __syncthreads();
  const int j = j0 + tx;
  if (j >= nb) return;
  const float lim = logf(static_cast<float>(min(kBlock, n - j * kBlock)));
#pragma unroll
  for (int rr = 0; rr < kTile / 8; ++rr) {
    const int il = ty * (kTile / 8) + rr, i = i0 + il;
    if (i >= nb) break;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int c = 0; c < D; ++c) acc[c & 3] = fmaf(sq[il][c], sk[tx][c], acc[c & 3]);
    const float v = half_s2 * ((acc[0] + acc[1]) + (acc[2] + acc[3]));
    const size_t o = (static_cast<size_t>(h) * nb + i) * nb + j;
    w[o] = (v > lim) ? 0.f : v;          // gated: the forward's spread
    if (wrank) wrank[o] = fminf(v, lim);  // clamped: the route's bonus
  }
}

}  // namespace

int launch_second_order(const void* q, const void* k, int in_bf16, int heads, int n, int d,
                        float scale, const float* kbar, float* qsq, float* kvar, float* w,
                        float* wrank, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  const dim3 g1(nb, heads);
  using BF = __nv_bfloat16;
  if (d == 128) {
    if (in_bf16)
      sq_var_kernel<BF, 128><<<g1, 128, 0, stream>>>(static_cast<const BF*>(q),
                                                     static_cast<const BF*>(k), kbar, n, nb, qsq, kvar);
    else
      sq_var_kernel<float, 128><<<g1, 128, 0, stream>>>(static_cast<const float*>(q),
                                                        static_cast<const float*>(k), kbar, n, nb,
                                                        qsq, kvar);
  } else {
    if (in_bf16)
      sq_var_kernel<BF, 64><<<g1, 64, 0, stream>>>(static_cast<const BF*>(q),
                                                   static_cast<const BF*>(k), kbar, n, nb, qsq, kvar);
    else
      sq_var_kernel<float, 64><<<g1, 64, 0, stream>>>(static_cast<const float*>(q),
                                                      static_cast<const float*>(k), kbar, n, nb,
                                                      qsq, kvar);
  }
  PISA_CHECK_LAUNCH();
  const dim3 g2(ceil_div(nb, kTile), ceil_div(nb, kTile), heads);
  const float half_s2 = 0.5f * scale * scale;
  if (d == 128)
    spread_kernel<128><<<g2, 256, 0, stream>>>(qsq, kvar, n, nb, half_s2, w, wrank);
  else
    spread_kernel<64><<<g2, 256, 0, stream>>>(qsq, kvar, n, nb, half_s2, w, wrank);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace pisa
