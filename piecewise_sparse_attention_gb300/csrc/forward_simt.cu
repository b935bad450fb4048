// Piecewise forward in float32 on the CUDA cores (float32 inputs; any
// supported head dim). "PISA: Piecewise Sparse Attention Is Wiser for
// Efficient Diffusion Transformers", Section 3.2, Eq. (3)-(6).
//
// One CTA per (query block, head), 256 threads: thread (r, p) owns query row
// r (0..63) and a quarter p of the key columns / output channels. Every key
// block j is visited once, in order, with one online softmax:
//   j in S_i : P = exp(e - m) on the exact logits e = s q.k;
//   j not in S_i : the block's centroid logit a = s q.kbar_j equals the mean of
//              its exact logits, and its first-order expansion contributes
//              P_n = exp(a - m) (1 + e_n - a) to the numerator and
//              n_j exp(a - m) to the denominator, which is
//              exp(a - m) (Vhat_j + q' H_j) and n_j exp(a - m) of Eq. (5)-(6).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
forward_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    int n, int nb, float scale, const int32_t* __restrict__ idx,
                    const int32_t* __restrict__ cnt, int max_sel, void* __restrict__ out,
                    int out_bf16, int32_t* dev_status, const float* __restrict__ spread) {
  constexpr int DP = D + 1;
  constexpr int CPT = D / 4;  // output channels per thread
  extern __shared__ float sm[];
  float* Qs = sm;                      // [64][DP]
  float* Ks = Qs + kBlock * DP;        // [64][DP]
  float* Vs = Ks + kBlock * DP;        // [64][D]
  float* Ps = Vs + kBlock * D;         // [64][65]
  uint32_t* sel = reinterpret_cast<uint32_t*>(Ps + kBlock * 65);  // [nwords]

  const int i = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  const int r = tid / 4, p = tid % 4;
  const int nwords = ceil_div(nb, 32);
  const size_t hoff = static_cast<size_t>(h) * n * D;
  const int qrow0 = i * kBlock;

  for (int w = tid; w < nwords; w += kThreads) sel[w] = 0u;
  for (int e = tid; e < kBlock * D; e += kThreads) {
    const int rr = e / D, c = e % D;
    Qs[rr * DP + c] = (qrow0 + rr < n) ? to_f(q[hoff + static_cast<size_t>(qrow0 + rr) * D + c]) : 0.f;
  }
  __syncthreads();
  {
    const int c = cnt[static_cast<size_t>(h) * nb + i];
    const int32_t* lst = idx + (static_cast<size_t>(h) * nb + i) * max_sel;
    for (int t = tid; t < min(c, max_sel); t += kThreads) {
      const int j = lst[t];
      if (j >= 0 && j < nb) atomicOr(&sel[j / 32], 1u << (j % 32));
      else report(dev_status, PISA_ERR_DEVICE_CHECK);
    }
  }

  float m = -INFINITY, l = 0.f;
  float o[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) o[c] = 0.f;

  for (int j = 0; j < nb; ++j) {
    __syncthreads();  // previous tile fully consumed
    const int krow0 = j * kBlock;
    const int nj = min(kBlock, n - krow0);
    for (int e = tid; e < kBlock * D; e += kThreads) {
      const int rr = e / D, c = e % D;
      const bool ok = rr < nj;
      const size_t g = hoff + static_cast<size_t>(krow0 + rr) * D + c;
      Ks[rr * DP + c] = ok ? to_f(k[g]) : 0.f;
      Vs[rr * D + c] = ok ? to_f(v[g]) : 0.f;
    }
    __syncthreads();
    const bool exact = (sel[j / 32] >> (j % 32)) & 1u;

    float e[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) e[u] = 0.f;
    for (int c = 0; c < D; ++c) {
      const float qc = Qs[r * DP + c];
#pragma unroll
      for (int u = 0; u < 16; ++u) e[u] = fmaf(qc, Ks[(p + 4 * u) * DP + c], e[u]);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) e[u] *= scale;

    float pv[16];
    if (exact) {
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (p + 4 * u < nj) mx = fmaxf(mx, e[u]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m, mx);
      const float corr = expf(m - mn);  // 0 on the first visited block
      float ls = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        pv[u] = (p + 4 * u < nj) ? expf(e[u] - mn) : 0.f;
        ls += pv[u];
      }
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      l = l * corr + ls;
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] *= corr;
      m = mn;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (p + 4 * u < nj) sum += e[u];
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      const float a = sum / static_cast<float>(nj);  // q'.kbar_j
      // second-order spread w_ij (optional) shifts the block's logit
      const float ae = spread ? a + spread[(static_cast<size_t>(h) * nb + i) * nb + j] : a;
      const float mn = fmaxf(m, ae);
      const float corr = expf(m - mn);
      const float alpha = expf(ae - mn);
#pragma unroll
      for (int u = 0; u < 16; ++u) pv[u] = (p + 4 * u < nj) ? alpha * (1.f + (e[u] - a)) : 0.f;
      l = l * corr + static_cast<float>(nj) * alpha;
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] *= corr;
      m = mn;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) Ps[r * 65 + p + 4 * u] = pv[u];
    __syncthreads();
    for (int kk = 0; kk < kBlock; ++kk) {
      const float pw = Ps[r * 65 + kk];
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] = fmaf(pw, Vs[kk * D + 4 * c + p], o[c]);
    }
  }

  const int row = qrow0 + r;
  if (row < n) {
    const float inv = 1.f / l;
    const size_t base = hoff + static_cast<size_t>(row) * D;
    if (out_bf16) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
#pragma unroll
      for (int c = 0; c < CPT; ++c) ob[base + 4 * c + p] = __float2bfloat16_rn(o[c] * inv);
    } else {
      float* of = static_cast<float*>(out);
#pragma unroll
      for (int c = 0; c < CPT; ++c) of[base + 4 * c + p] = o[c] * inv;
    }
  }
}

}  // namespace

int launch_forward_simt(const void* q, const void* k, const void* v, int heads,
                        int n, int d, float scale, const int32_t* idx, const int32_t* cnt,
                        int max_sel, void* out, int out_bf16, int32_t* dev_status,
                        cudaStream_t stream, const float* spread) {
  const int nb = ceil_div(n, kBlock);
  const size_t smem = (2 * kBlock * (d + 1) + kBlock * d + kBlock * 65) * sizeof(float) +
                      ceil_div(nb, 32) * sizeof(uint32_t);
  dim3 grid(nb, heads);
  auto run = [&](auto kern, auto tag) -> int {
    using T = decltype(tag);
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)));
    kern<<<grid, kThreads, smem, stream>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                           static_cast<const T*>(v), n, nb, scale, idx, cnt,
                                           max_sel, out, out_bf16, dev_status, spread);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  return d == 128 ? run(forward_simt_kernel<float, 128>, 0.f)
                  : run(forward_simt_kernel<float, 64>, 0.f);
}

}  // namespace pisa

// ---------------------------------------------------------------------------
// Hybrid-order forward ("PISA", Section 3.3 Eq. 9-10), float32 CUDA cores.
//   exact phase:   j in S_i, as above (exp on the exact logits);
//   zeroth order:  j not in S_i, alpha = exp(q'.kbar_j - m): l += n_j alpha,
//                  O += alpha Vhat_j, tail += alpha;
//   first order:   O += tail (q' Hbar) with the query-independent Hbar.
// ---------------------------------------------------------------------------
namespace pisa {
namespace {

constexpr int kHThreads = 256;
constexpr int kChunk = 32;  // centroid rows staged per step

template <typename T, int D>
__global__ void __launch_bounds__(kHThreads)
forward_hybrid_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                           const T* __restrict__ v, int n, int nb, float scale,
                           const float* __restrict__ kbar, const float* __restrict__ vsum,
                           const float* __restrict__ hbar, const int32_t* __restrict__ idx,
                           const int32_t* __restrict__ cnt, int max_sel, void* __restrict__ out,
                           int out_bf16, int32_t* dev_status) {
  constexpr int DP = D + 1;
  constexpr int CPT = D / 4;
  extern __shared__ float sm[];
  float* Qs = sm;                   // [64][DP]
  float* Ks = Qs + kBlock * DP;     // [64][DP]   (later: centroid chunk, then Hbar)
  float* Vs = Ks + kBlock * DP;     // [64][D]
  float* Ps = Vs + kBlock * D;      // [64][65]
  uint32_t* sel = reinterpret_cast<uint32_t*>(Ps + kBlock * 65);

  const int i = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x;
  const int r = tid / 4, p = tid % 4;
  const int nwords = ceil_div(nb, 32);
  const size_t hoff = static_cast<size_t>(h) * n * D;
  const int qrow0 = i * kBlock;

  for (int w = tid; w < nwords; w += kHThreads) sel[w] = 0u;
  for (int e = tid; e < kBlock * D; e += kHThreads) {
    const int rr = e / D, c = e % D;
    Qs[rr * DP + c] =
        (qrow0 + rr < n) ? to_f(q[hoff + static_cast<size_t>(qrow0 + rr) * D + c]) : 0.f;
  }
  __syncthreads();
  const int c_sel = min(cnt[static_cast<size_t>(h) * nb + i], max_sel);
  const int32_t* lst = idx + (static_cast<size_t>(h) * nb + i) * max_sel;
  for (int t = tid; t < c_sel; t += kHThreads) {
    const int j = lst[t];
    if (j >= 0 && j < nb) atomicOr(&sel[j / 32], 1u << (j % 32));
    else report(dev_status, PISA_ERR_DEVICE_CHECK);
  }
  __syncthreads();

  float m = -INFINITY, l = 0.f, tail = 0.f;
  float o[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) o[c] = 0.f;

  // ---- exact phase over S_i ----
  for (int t = 0; t < c_sel; ++t) {
    const int j = lst[t];
    if (j < 0 || j >= nb) continue;
    __syncthreads();
    const int krow0 = j * kBlock;
    const int nj = min(kBlock, n - krow0);
    for (int e = tid; e < kBlock * D; e += kHThreads) {
      const int rr = e / D, c = e % D;
      const bool ok = rr < nj;
      const size_t g = hoff + static_cast<size_t>(krow0 + rr) * D + c;
      Ks[rr * DP + c] = ok ? to_f(k[g]) : 0.f;
      Vs[rr * D + c] = ok ? to_f(v[g]) : 0.f;
    }
    __syncthreads();
    float e[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) e[u] = 0.f;
    for (int c = 0; c < D; ++c) {
      const float qc = Qs[r * DP + c];
#pragma unroll
      for (int u = 0; u < 16; ++u) e[u] = fmaf(qc, Ks[(p + 4 * u) * DP + c], e[u]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      e[u] *= scale;
      if (p + 4 * u < nj) mx = fmaxf(mx, e[u]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    const float corr = expf(m - mn);
    float pv[16], ls = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      pv[u] = (p + 4 * u < nj) ? expf(e[u] - mn) : 0.f;
      ls += pv[u];
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    l = l * corr + ls;
    tail *= corr;
#pragma unroll
    for (int c = 0; c < CPT; ++c) o[c] *= corr;
    m = mn;
#pragma unroll
    for (int u = 0; u < 16; ++u) Ps[r * 65 + p + 4 * u] = pv[u];
    __syncthreads();
    for (int kk = 0; kk < kBlock; ++kk) {
      const float pw = Ps[r * 65 + kk];
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] = fmaf(pw, Vs[kk * D + 4 * c + p], o[c]);
    }
  }

  // ---- zeroth order over the remaining blocks, in chunks of centroids ----
  float* Cs = Ks;  // [kChunk][DP] centroids
  float* Ws = Vs;  // [kChunk][D]  value sums
  const float* kbh = kbar + static_cast<size_t>(h) * nb * D;
  const float* vsh = vsum + static_cast<size_t>(h) * nb * D;
  for (int j0 = 0; j0 < nb; j0 += kChunk) {
    const int cn = min(kChunk, nb - j0);
    __syncthreads();
    for (int e = tid; e < kChunk * D; e += kHThreads) {
      const int rr = e / D, c = e % D;
      const bool ok = rr < cn;
      Cs[rr * DP + c] = ok ? kbh[static_cast<size_t>(j0 + rr) * D + c] : 0.f;
      Ws[rr * D + c] = ok ? vsh[static_cast<size_t>(j0 + rr) * D + c] : 0.f;
    }
    __syncthreads();
    // centroid logits of this chunk: thread (r, p) sums channels p, p+4, ...
    float a[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) a[u] = 0.f;
    for (int c = p; c < D; c += 4) {
      const float qc = Qs[r * DP + c];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) a[u] = fmaf(qc, Cs[u * DP + c], a[u]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      a[u] += __shfl_xor_sync(0xffffffffu, a[u], 1);
      a[u] += __shfl_xor_sync(0xffffffffu, a[u], 2);
      a[u] *= scale;
      const int j = j0 + u;
      const bool use = u < cn && !((sel[j >> 5] >> (j & 31)) & 1u);
      if (use) mx = fmaxf(mx, a[u]);
    }
    // (mx stays -inf only when every block of the chunk is exact; the route is
    // shared by all rows of the CTA, so the branch is uniform)
    if (mx != -INFINITY) {
      const float mn = fmaxf(m, mx);
      const float corr = expf(m - mn);
      l *= corr;
      tail *= corr;
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] *= corr;
      m = mn;
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const int j = j0 + u;
        const bool use = u < cn && !((sel[j >> 5] >> (j & 31)) & 1u);
        if (use) {
          const float al = expf(a[u] - m);
          const int nj = min(kBlock, n - j * kBlock);
          l = fmaf(static_cast<float>(nj), al, l);
          tail += al;
#pragma unroll
          for (int c = 0; c < CPT; ++c) o[c] = fmaf(al, Ws[u * D + 4 * c + p], o[c]);
        }
      }
    }
  }

  // ---- global first order: O += tail (q' Hbar) ----
  __syncthreads();
  float* Hs = Ks;  // Hbar rows staged in two halves of D/2 rows
  const float* hb = hbar + static_cast<size_t>(h) * D * D;
  for (int half = 0; half < 2; ++half) {
    __syncthreads();
    for (int e = tid; e < (D / 2) * D; e += kHThreads) Hs[e] = hb[static_cast<size_t>(half) * (D / 2) * D + e];
    __syncthreads();
    for (int cr = 0; cr < D / 2; ++cr) {
      const float qc = scale * Qs[r * DP + half * (D / 2) + cr] * tail;
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[c] = fmaf(qc, Hs[cr * D + 4 * c + p], o[c]);
    }
  }

  const int row = qrow0 + r;
  if (row < n) {
    const float inv = 1.f / l;
    const size_t base = hoff + static_cast<size_t>(row) * D;
    if (out_bf16) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
#pragma unroll
      for (int c = 0; c < CPT; ++c) ob[base + 4 * c + p] = __float2bfloat16_rn(o[c] * inv);
    } else {
      float* of = static_cast<float*>(out);
#pragma unroll
      for (int c = 0; c < CPT; ++c) of[base + 4 * c + p] = o[c] * inv;
    }
  }
}

}  // namespace

int launch_forward_hybrid_simt(const void* q, const void* k, const void* v,
                               int heads, int n, int d, float scale, const float* kbar,
                               const float* vsum, const float* hbar, const int32_t* idx,
                               const int32_t* cnt, int max_sel, void* out, int out_bf16,
                               int32_t* dev_status, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  const size_t smem = (2 * kBlock * (d + 1) + kBlock * d + kBlock * 65) * sizeof(float) +
                      ceil_div(nb, 32) * sizeof(uint32_t);
  dim3 grid(nb, heads);
  auto run = [&](auto kern, auto tag) -> int {
    using T = decltype(tag);
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
    kern<<<grid, kHThreads, smem, stream>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                            static_cast<const T*>(v), n, nb, scale, kbar, vsum,
                                            hbar, idx, cnt, max_sel, out, out_bf16, dev_status);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  return d == 128 ? run(forward_hybrid_simt_kernel<float, 128>, 0.f)
                  : run(forward_hybrid_simt_kernel<float, 64>, 0.f);
}

}  // namespace pisa
