// Block statistics: qbar_j, kbar_j (means), Vhat_j (sum) and optionally
// H_j = sum_n (k_{j,n} - kbar_j)^T v_{j,n}.
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Section 3.2 "Formulation" and Eq. (5)-(6), Appendix C
// "Notation", Figure 4 "Prepare Phase".
//
// One CTA of 256 threads per (block, head). Rows are read as 16-byte chunks so
// that a warp covers two (d=128 bf16) or more full rows per load: every load
// instruction is fully coalesced. Means and sums use compensated float32
// accumulation (TwoSum) and are rounded once, so the routing scores computed
// from them see at most one rounding of the exact block mean.
#include "common.cuh"
#include "kernels.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;

template <typename T, int D, bool WITH_H>
__global__ void __launch_bounds__(kThreads)
block_stats_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   int n, int nb, float* __restrict__ qbar, float* __restrict__ kbar,
                   float* __restrict__ vsum, void* __restrict__ hmat, int h_bf16) {
  constexpr int CH = Chunk<T>::kElems;     // channels per 16-byte chunk
  constexpr int NCHUNK = D / CH;           // chunks per row
  constexpr int NG = kThreads / NCHUNK;    // row groups
  constexpr int RPT = kBlock / NG;         // rows per thread
  static_assert(RPT * NG == kBlock, "layout");

  extern __shared__ float smem[];
  // partial sums: [NG][D] for s and for c
  float* ps = smem;
  float* pc = smem + NG * D;
  float* kt = smem + 2 * NG * D;          // [64][D+1] centred keys (WITH_H)
  float* vt = kt + kBlock * (D + 1);      // [64][D+1] values (WITH_H)
  __shared__ float s_mean[D];

  const int j = blockIdx.x;
  const int h = blockIdx.y;
  const int row0 = j * kBlock;
  const int nj = min(kBlock, n - row0);
  const int tid = threadIdx.x;
  const int chunk = tid % NCHUNK;
  const int grp = tid / NCHUNK;
  const size_t head_off = static_cast<size_t>(h) * n * D;
  const size_t out_off = (static_cast<size_t>(h) * nb + j) * D;

  const T* srcs[3] = {q, k, v};
  float* dsts[3] = {qbar, kbar, vsum};
#pragma unroll 1
  for (int which = 0; which < 3; ++which) {
    float* dst = dsts[which];
    const bool need_tile = WITH_H && which >= 1;
    if (dst == nullptr && !need_tile && !(WITH_H && which == 1)) continue;
    const T* src = srcs[which] + head_off;
    CSum acc[CH];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int row = grp + r * NG;
      if (row < nj) {
        float f[CH];
        Chunk<T>::load(src + static_cast<size_t>(row0 + row) * D + chunk * CH, f);
#pragma unroll
        for (int c = 0; c < CH; ++c) acc[c].add(f[c]);
        if (need_tile) {
          float* tile = (which == 1) ? kt : vt;
#pragma unroll
          for (int c = 0; c < CH; ++c) tile[row * (D + 1) + chunk * CH + c] = f[c];
        }
      }
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      ps[grp * D + chunk * CH + c] = acc[c].s;
      pc[grp * D + chunk * CH + c] = acc[c].c;
    }
    __syncthreads();
    if (tid < D) {
      CSum tot;
      for (int g = 0; g < NG; ++g) {
        CSum part;
        part.s = ps[g * D + tid];
        part.c = pc[g * D + tid];
        tot.merge(part);
      }
      const float sum = tot.value();
      const float res = (which == 2) ? sum : __fdiv_rn(sum, static_cast<float>(nj));
      if (dst != nullptr) dst[out_off + tid] = res;
      if (which == 1) s_mean[tid] = res;
    }
    __syncthreads();
  }

  if constexpr (WITH_H) {
    // centre the staged keys, zero rows past the end of a partial block
    for (int e = tid; e < kBlock * D; e += kThreads) {
      const int row = e / D, c = e % D;
      const bool ok = row < nj;
      kt[row * (D + 1) + c] = ok ? __fsub_rn(kt[row * (D + 1) + c], s_mean[c]) : 0.f;
      if (!ok) vt[row * (D + 1) + c] = 0.f;
    }
    __syncthreads();
    // H[c][e]: each thread owns a TC x TE sub-tile
    constexpr int TILE = (D == 128) ? 8 : 4;
    constexpr int PER_ROW = D / TILE;
    const int c0 = (tid / PER_ROW) * TILE;
    const int e0 = (tid % PER_ROW) * TILE;
    float accH[TILE][TILE];
#pragma unroll
    for (int a = 0; a < TILE; ++a)
#pragma unroll
      for (int b = 0; b < TILE; ++b) accH[a][b] = 0.f;
    for (int r = 0; r < kBlock; ++r) {
      float kc[TILE], vv[TILE];
#pragma unroll
      for (int a = 0; a < TILE; ++a) kc[a] = kt[r * (D + 1) + c0 + a];
#pragma unroll
      for (int b = 0; b < TILE; ++b) vv[b] = vt[r * (D + 1) + e0 + b];
#pragma unroll
      for (int a = 0; a < TILE; ++a)
#pragma unroll
        for (int b = 0; b < TILE; ++b) accH[a][b] = __fmaf_rn(kc[a], vv[b], accH[a][b]);
    }
    const size_t hbase = ((static_cast<size_t>(h) * nb + j) * D) * D;
    if (h_bf16) {
      __nv_bfloat16* H = static_cast<__nv_bfloat16*>(hmat) + hbase;
#pragma unroll
      for (int a = 0; a < TILE; ++a)
#pragma unroll
        for (int b = 0; b < TILE; ++b)
          H[static_cast<size_t>(c0 + a) * D + e0 + b] = __float2bfloat16_rn(accH[a][b]);
    } else {
      float* H = static_cast<float*>(hmat) + hbase;
#pragma unroll
      for (int a = 0; a < TILE; ++a)
#pragma unroll
        for (int b = 0; b < TILE; ++b) H[static_cast<size_t>(c0 + a) * D + e0 + b] = accH[a][b];
    }
  }
}

template <typename T, int D, bool WITH_H>
int launch(const void* q, const void* k, const void* v, int heads, int n, float* qbar,
           float* kbar, float* vsum, void* hmat, int h_bf16, cudaStream_t stream) {
  constexpr int CH = Chunk<T>::kElems;
  constexpr int NG = kThreads / (D / CH);
  const int nb = ceil_div(n, kBlock);
  size_t smem = 2 * NG * D * sizeof(float);
  if (WITH_H) smem += 2 * kBlock * (D + 1) * sizeof(float);
  auto kern = block_stats_kernel<T, D, WITH_H>;
  if (smem > 48 * 1024) {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)));
  }
  dim3 grid(nb, heads);
  kern<<<grid, kThreads, smem, stream>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                         static_cast<const T*>(v), n, nb, qbar, kbar, vsum,
                                         hmat, h_bf16);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace

int launch_block_stats(const void* q, const void* k, const void* v, int in_bf16, int heads,
                       int n, int d, float* qbar, float* kbar, float* vsum, void* hmat,
                       int h_bf16, cudaStream_t stream) {
  const bool wh = hmat != nullptr;
#define PISA_STATS_CASE(T, D)                                                                  \
  return wh ? launch<T, D, true>(q, k, v, heads, n, qbar, kbar, vsum, hmat, h_bf16, stream)    \
            : launch<T, D, false>(q, k, v, heads, n, qbar, kbar, vsum, hmat, h_bf16, stream)
  if (in_bf16) {
    if (d == 128) PISA_STATS_CASE(__nv_bfloat16, 128);
    PISA_STATS_CASE(__nv_bfloat16, 64);
  } else {
    if (d == 128) PISA_STATS_CASE(float, 128);
    PISA_STATS_CASE(float, 64);
  }
#undef PISA_STATS_CASE
}

}  // namespace pisa
