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
// sq_var_kernel: one CTA per (block, head), 16-byte row chunks with several
//   rows in flight, float32 sums reduced over the row groups in shared memory;
// spread_kernel: 64 x 64 tiles of w per CTA, 4 x 4 float32 outputs a thread
//   over d from channel-major shared tiles, then the gate.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

constexpr int kSqThreads = 128;

// One CTA per (block, head). Rows are read in 16-byte chunks: CPR chunks per
// row, RPP rows per pass, each thread summing its chunk's channels over the
// rows of its row group; the row groups are then summed through shared memory.
template <typename T, int D>
__global__ void __launch_bounds__(kSqThreads)
sq_var_kernel(const T* __restrict__ q, const T* __restrict__ k, const float* __restrict__ kbar,
              int n, int nb, float* __restrict__ qsq, float* __restrict__ kvar) {
  constexpr int E = Chunk<T>::kElems;   // channels per 16-byte chunk
  constexpr int CPR = D / E;            // chunks per row
  constexpr int RPP = kSqThreads / CPR; // rows per pass
  __shared__ float sq[RPP][D];
  __shared__ float sk[RPP][D];
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int ch = tid % CPR, rg = tid / CPR, c0 = ch * E;
  const int r0 = j * kBlock, nj = min(kBlock, n - r0);
  const size_t base = (static_cast<size_t>(h) * n + r0) * D + c0;
  const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D + c0;
  float kbv[E], qs[E], ks[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kbv[e] = kb[e];
    qs[e] = ks[e] = 0.f;
  }
#pragma unroll 4
  for (int r = rg; r < nj; r += RPP) {
    float fq[E], fk[E];
    Chunk<T>::load(q + base + static_cast<size_t>(r) * D, fq);
    Chunk<T>::load(k + base + static_cast<size_t>(r) * D, fk);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qs[e] = fmaf(fq[e], fq[e], qs[e]);
      const float y = fk[e] - kbv[e];
      ks[e] = fmaf(y, y, ks[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    sq[rg][c0 + e] = qs[e];
    sk[rg][c0 + e] = ks[e];
  }
  __syncthreads();
  const float inv = 1.f / static_cast<float>(nj);
  for (int c = tid; c < D; c += kSqThreads) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int g = 0; g < RPP; ++g) {
      a += sq[g][c];
      b += sk[g][c];
    }
    const size_t o = (static_cast<size_t>(h) * nb + j) * D + c;
    qsq[o] = a * inv;
    kvar[o] = b * inv;
  }
}

constexpr int kTile = 64;     // w tile edge
constexpr int kSpThreads = 256;

// 64 x 64 tile of w per CTA, 4 x 4 outputs per thread; qsq and kvar of the
// tile's blocks staged channel-major in shared memory (row stride 65 floats),
// so each channel step is two 16-byte loads for 16 FMAs.
template <int D>
__global__ void __launch_bounds__(kSpThreads)
spread_kernel(const float* __restrict__ qsq, const float* __restrict__ kvar, int n, int nb,
              float half_s2, float* __restrict__ w, float* __restrict__ wrank) {
  constexpr int LDT = kTile + 4;  // 16-byte aligned rows, staggered banks
  extern __shared__ __align__(16) float smem[];
  float* sq = smem;               // [D][LDT]: sq[c][i] = qsq[i0 + i][c]
  float* sk = smem + D * LDT;     // [D][LDT]: sk[c][j] = kvar[j0 + j][c]
  const int h = blockIdx.z, i0 = blockIdx.y * kTile, j0 = blockIdx.x * kTile;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  // consecutive threads take consecutive rows: the transposing stores then
  // fall on consecutive banks
  for (int e = tid; e < kTile * (D / 4); e += kSpThreads) {
    const int r = e % kTile, c = (e / kTile) * 4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (i0 + r < nb) a = __ldg(reinterpret_cast<const float4*>(qsq + (static_cast<size_t>(h) * nb + i0 + r) * D + c));
    if (j0 + r < nb) b = __ldg(reinterpret_cast<const float4*>(kvar + (static_cast<size_t>(h) * nb + j0 + r) * D + c));
    sq[(c + 0) * LDT + r] = a.x;
    sq[(c + 1) * LDT + r] = a.y;
    sq[(c + 2) * LDT + r] = a.z;
    sq[(c + 3) * LDT + r] = a.w;
    sk[(c + 0) * LDT + r] = b.x;
    sk[(c + 1) * LDT + r] = b.y;
    sk[(c + 2) * LDT + r] = b.z;
    sk[(c + 3) * LDT + r] = b.w;
  }
  __syncthreads();
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int c = 0; c < D; ++c) {
    const float4 x = *reinterpret_cast<const float4*>(sq + c * LDT + 4 * ty);
    const float4 y = *reinterpret_cast<const float4*>(sk + c * LDT + 4 * tx);
    const float xa[4] = {x.x, x.y, x.z, x.w}, yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], yb[b], acc[a][b]);
  }
  float lim[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int j = j0 + 4 * tx + b;
    lim[b] = (j < nb) ? logf(static_cast<float>(min(kBlock, n - j * kBlock))) : 0.f;
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = i0 + 4 * ty + a;
    if (i >= nb) break;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = j0 + 4 * tx + b;
      if (j >= nb) break;
      const float v = half_s2 * acc[a][b];
      const size_t o = (static_cast<size_t>(h) * nb + i) * nb + j;
      w[o] = (v > lim[b]) ? 0.f : v;           // gated: the forward's spread
      if (wrank) wrank[o] = fminf(v, lim[b]);  // clamped: the route's bonus
    }
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
      sq_var_kernel<BF, 128><<<g1, kSqThreads, 0, stream>>>(static_cast<const BF*>(q),
                                                            static_cast<const BF*>(k), kbar, n, nb,
                                                            qsq, kvar);
    else
      sq_var_kernel<float, 128><<<g1, kSqThreads, 0, stream>>>(static_cast<const float*>(q),
                                                               static_cast<const float*>(k), kbar,
                                                               n, nb, qsq, kvar);
  } else {
    if (in_bf16)
      sq_var_kernel<BF, 64><<<g1, kSqThreads, 0, stream>>>(static_cast<const BF*>(q),
                                                           static_cast<const BF*>(k), kbar, n, nb,
                                                           qsq, kvar);
    else
      sq_var_kernel<float, 64><<<g1, kSqThreads, 0, stream>>>(static_cast<const float*>(q),
                                                              static_cast<const float*>(k), kbar,
                                                              n, nb, qsq, kvar);
  }
  PISA_CHECK_LAUNCH();
  const dim3 g2(ceil_div(nb, kTile), ceil_div(nb, kTile), heads);
  const float half_s2 = 0.5f * scale * scale;
  if (d == 128) {
    const int sm = 2 * 128 * (kTile + 4) * 4;
    PISA_CUDA_TRY(cudaFuncSetAttribute(spread_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sm));
    spread_kernel<128><<<g2, kSpThreads, sm, stream>>>(qsq, kvar, n, nb, half_s2, w, wrank);
  } else {
    const int sm = 2 * 64 * (kTile + 4) * 4;
    spread_kernel<64><<<g2, kSpThreads, sm, stream>>>(qsq, kvar, n, nb, half_s2, w, wrank);
  }
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace pisa
