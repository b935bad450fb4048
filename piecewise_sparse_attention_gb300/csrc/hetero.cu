// Per-block heterogeneity of the first-order statistics,
//   M_j = || H_j - Hbar ||,   H_j = sum_n (k_{j,n} - kbar_j)^T v_{j,n},
// the prior of the covariance-aware block selection ("PISA: Piecewise Sparse
// Attention Is Wiser for Efficient Diffusion Transformers", Section 3.3
// "Covariance-Aware Block Selection", Eq. 11, with the norm of Theorem 3.1;
// Appendix D). Two norms:
//   spectral  - the largest singular value (the norm Section 3.3 writes);
//   Frobenius - the root of the sum of squares (the Piecewise-Taylor-Attention
//               README's router).
//
// One CTA (256 threads) per (block, head):
//   1. the block's centred keys and values go to shared memory as float32;
//   2. A = Kc^T V - Hbar, one 8x8 (d = 128) or 4x4 (d = 64) register tile per
//      thread; Frobenius: sum of squares, reduced in double, done;
//   3. spectral: M_j^2 = lambda_max(A^T A) by the Lanczos iteration on
//      A^T A applied as A^T (A q) to the register tiles (A^T A is never
//      formed), with full reorthogonalisation, stopped on the residual of the
//      top Ritz pair (relative 1e-7; at most d steps, where the Krylov space
//      is the whole space); the top Ritz value of the tridiagonal by
//      Sturm-count multisection on each warp.
// Everything is float32 except the Frobenius reduction. The Ritz values are
// lower bounds of lambda_max that converge to it; on the workloads' blocks the
// stop comes after 8 to 28 steps.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

constexpr int kThreads = 256;

template <int D>
struct HeteroSmem {
  static constexpr int KV = 2 * kBlock * D;  // centred keys and values, float32
  static constexpr int BASIS = D * D;        // Lanczos vectors (after the K/V phase)
  static constexpr int BIG = KV > BASIS ? KV : BASIS;
  // per-warp partials [8][D], Gram-Schmidt coefficients [2][D], per-warp alpha,
  // beta, beta^2 [8][3][D]
  static constexpr int VEC = (8 + 2 + 8 * 3) * D;
  static constexpr size_t bytes(bool spectral) {
    return spectral ? static_cast<size_t>(BIG + VEC) * 4 : static_cast<size_t>(KV) * 4 + 64;
  }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int D, bool SPECTRAL>
__global__ void __launch_bounds__(kThreads)
hetero_kernel(const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ kbar,
              const float* __restrict__ hbar, int n, int nb, float* __restrict__ mnorm) {
  using S = HeteroSmem<D>;
  constexpr int CH = Chunk<T>::kElems;
  constexpr int TL = D / 16;  // register tile edge
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;                // [64][D] centred keys
  float* sV = sm + kBlock * D;   // [64][D] values
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int r0 = j * kBlock;
  const int nj = min(kBlock, n - r0);

  // ---- 1. centred keys and values of block j ---------------------------------
  const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D;
  const size_t base = (static_cast<size_t>(h) * n + r0) * D;
  for (int e = tid; e < kBlock * (D / CH); e += kThreads) {
    const int row = e / (D / CH), c0 = (e % (D / CH)) * CH;
    float fk[CH], fv[CH];
    if (row < nj) {
      Chunk<T>::load(k + base + static_cast<size_t>(row) * D + c0, fk);
      Chunk<T>::load(v + base + static_cast<size_t>(row) * D + c0, fv);
#pragma unroll
      for (int i = 0; i < CH; ++i) fk[i] -= kb[c0 + i];
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i) fk[i] = fv[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      sK[row * D + c0 + i] = fk[i];
      sV[row * D + c0 + i] = fv[i];
    }
  }
  __syncthreads();

  // ---- 2. A = Kc^T V - Hbar, rows ty*TL.., columns tx*TL.. of this thread -----
  const int ty = tid / 16, tx = tid % 16;
  float acc[TL][TL];
#pragma unroll
  for (int a = 0; a < TL; ++a)
#pragma unroll
    for (int b = 0; b < TL; ++b) acc[a][b] = 0.f;
#pragma unroll 4
  for (int t = 0; t < kBlock; ++t) {
    float ka[TL], vb[TL];
#pragma unroll
    for (int a = 0; a < TL; ++a) {
      ka[a] = sK[t * D + ty * TL + a];
      vb[a] = sV[t * D + tx * TL + a];
    }
#pragma unroll
    for (int a = 0; a < TL; ++a)
#pragma unroll
      for (int b = 0; b < TL; ++b) acc[a][b] = fmaf(ka[a], vb[b], acc[a][b]);
  }
  const float* hb = hbar + static_cast<size_t>(h) * D * D;
#pragma unroll
  for (int a = 0; a < TL; ++a)
#pragma unroll
    for (int b = 0; b < TL; ++b) acc[a][b] -= hb[(ty * TL + a) * D + tx * TL + b];

  __shared__ double s_part[kThreads / 32];
  if (!SPECTRAL) {
    float sq = 0.f;
#pragma unroll
    for (int a = 0; a < TL; ++a)
#pragma unroll
      for (int b = 0; b < TL; ++b) sq = fmaf(acc[a][b], acc[a][b], sq);
    const double w = warp_sum_d(static_cast<double>(sq));
    if (lane == 0) s_part[warp] = w;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int i = 0; i < kThreads / 32; ++i) t += s_part[i];
      mnorm[static_cast<size_t>(h) * nb + j] = static_cast<float>(sqrt(t));
    }
    return;
  }

  // ---- 3. spectral norm: Lanczos on C = A^T A -----------------------------------
  // q_0 fixed and dense; step k: w = A^T (A q_k), two classical Gram-Schmidt
  // passes against q_0..q_k (full reorthogonalisation; the first pass also
  // removes beta_{k-1} q_{k-1}), alpha_k = q_k.(A^T A q_k), beta_k = |w|,
  // q_{k+1} = w / beta_k. The Ritz values of the tridiagonal T_m (diagonal
  // alpha, off-diagonal beta) are lower bounds of lambda_max(C) that converge
  // to it; every 4 steps the largest one, theta, is located by Sturm-count
  // multisection, and the step stops once the residual of its Ritz vector,
  // beta_{m-1} |y_{m-1}| (y the normalised eigenvector of T_m), is below
  // 1e-7 theta: theta is then within 1e-7 theta of an eigenvalue of C. At
  // m = D the Krylov space is the whole space and theta is the answer.
  __syncthreads();  // every read of sK / sV is done before the basis overwrites them
  constexpr int VPL = D / 32;                    // vector elements per lane: VPL*lane ..
  float* basis = sm;                             // [D][D] q_0, q_1, ... one per row
  float* part = sm + S::BIG;                     // [8][D] per-warp partial A^T (A q)
  float* hdot = part + 8 * D;                    // [2][D] Gram-Schmidt coefficients
  float* wal = hdot + 2 * D + warp * 3 * D;      // this warp's copy of alpha [D],
  float* wbe = wal + D;                          //   beta [D]
  float* wb2 = wbe + D;                          //   and beta^2 [D]
  const int c0 = tx * TL;

  float q[VPL];  // this lane's elements of q_k (every warp holds all of q_k)
  {
    float ss = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      const uint32_t e = static_cast<uint32_t>(VPL * lane + x);
      const uint32_t hsh = (e + 1u) * 2654435761u;
      q[x] = 0.25f + static_cast<float>(hsh >> 8) * (1.f / 16777216.f);  // in [0.25, 1.25)
      q[x] = (hsh & 1u) ? -q[x] : q[x];
      ss = fmaf(q[x], q[x], ss);
    }
    const float inv = rsqrtf(warp_sum(ss));
#pragma unroll
    for (int x = 0; x < VPL; ++x) q[x] *= inv;
    if (warp == 0) {
#pragma unroll
      for (int x = 0; x < VPL; ++x) basis[VPL * lane + x] = q[x];
    }
  }
  float theta = 0.f;
  for (int k = 0; k < D; ++k) {
    // u = A q_k on this thread's rows (sum over the 16 column threads of a row group)
    float qv[TL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      qv[x] = __shfl_sync(0xffffffffu, q[x], 2 * tx);
      qv[VPL + x] = __shfl_sync(0xffffffffu, q[x], 2 * tx + 1);
    }
    float u[TL];
#pragma unroll
    for (int a = 0; a < TL; ++a) {
      float t = 0.f;
#pragma unroll
      for (int b = 0; b < TL; ++b) t = fmaf(acc[a][b], qv[b], t);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      u[a] = t;
    }
    // this thread's part of A^T u: its rows, its columns; the warp's two row groups summed
#pragma unroll
    for (int b = 0; b < TL; ++b) {
      float t = 0.f;
#pragma unroll
      for (int a = 0; a < TL; ++a) t = fmaf(acc[a][b], u[a], t);
      t += __shfl_xor_sync(0xffffffffu, t, 16);
      if (lane < 16) part[warp * D + c0 + b] = t;
    }
    __syncthreads();
    float w[VPL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      float t = 0.f;
#pragma unroll
      for (int p = 0; p < kThreads / 32; ++p) t += part[p * D + VPL * lane + x];
      w[x] = t;
    }
    float alpha = 0.f;
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      float* hd = hdot + ps * D;
      for (int i = warp; i <= k; i += kThreads / 32) {
        float t = 0.f;
#pragma unroll
        for (int x = 0; x < VPL; ++x) t = fmaf(basis[i * D + VPL * lane + x], w[x], t);
        t = warp_sum(t);
        if (lane == 0) hd[i] = t;
      }
      __syncthreads();
      for (int i = 0; i <= k; ++i) {
        const float hc = hd[i];
#pragma unroll
        for (int x = 0; x < VPL; ++x) w[x] = fmaf(-hc, basis[i * D + VPL * lane + x], w[x]);
      }
      alpha += hd[k];
    }
    float ss = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) ss = fmaf(w[x], w[x], ss);
    const float beta = sqrtf(warp_sum(ss));
    if (lane == 0) {
      wal[k] = alpha;
      wbe[k] = beta;
      wb2[k] = beta * beta;
    }
    __syncwarp();
    const int m = k + 1;
    if (beta == 0.f || m % 4 == 0 || m == D) {
      // theta = largest eigenvalue of T_m: Gershgorin interval, 32 trial
      // points per round (lane l tests lo + (l + 1)(hi - lo) / 33)
      float lo = theta, hi = 0.f;
      for (int i = lane; i < m; i += 32) {
        const float r = (i > 0 ? wbe[i - 1] : 0.f) + (i < m - 1 ? wbe[i] : 0.f);
        hi = fmaxf(hi, wal[i] + r);
      }
      hi = warp_max(hi);
      hi = hi * 1.000001f;
      lo = fminf(lo, hi);
      const float tiny = fmaxf(1e-30f * hi, 1e-36f);
      for (int round = 0; round < 12 && hi - lo > 1e-7f * hi; ++round) {
        const float mu = lo + (hi - lo) * static_cast<float>(lane + 1) * (1.f / 33.f);
        int below = 0;
        float qd = wal[0] - mu;
        below += qd < 0.f;
        for (int i = 1; i < m; ++i) {
          if (fabsf(qd) < tiny) qd = -tiny;
          qd = wal[i] - mu - __fdividef(wb2[i - 1], qd);
          below += qd < 0.f;
        }
        const unsigned all = __ballot_sync(0xffffffffu, below == m);  // lambda_max < mu
        const int f = all ? __ffs(all) - 1 : 32;
        const float new_hi = (f < 32) ? __shfl_sync(0xffffffffu, mu, f & 31) : hi;
        const float new_lo = (f > 0) ? __shfl_sync(0xffffffffu, mu, (f - 1) & 31) : lo;
        hi = new_hi;
        lo = new_lo;
      }
      theta = 0.5f * (lo + hi);
      // last component y_{m-1} of the normalised eigenvector of T_m, from the
      // bottom up (the stable direction: a converging Ritz vector decays
      // towards the end of the basis): x_{m-1} = 1, |x_i| = |x_{i+1}| |e_{i+1}|
      // / beta_i with e the pivots of the trailing blocks of T_m - hi I
      float xc = 1.f, xs = 1.f, xl = 1.f, e = wal[m - 1] - hi;
      for (int i = m - 2; i >= 0; --i) {
        xc = (wbe[i] > 0.f) ? xc * fabsf(e) / wbe[i] : 0.f;
        if (xc > 1e18f) {
          xc *= 1e-18f;
          xs *= 1e-36f;
          xl *= 1e-18f;
        }
        xs = fmaf(xc, xc, xs);
        if (fabsf(e) < tiny) e = -tiny;
        e = wal[i] - hi - __fdividef(wb2[i], e);
      }
      const float resid = beta * xl * rsqrtf(xs);
      if (beta == 0.f || resid <= 1e-7f * fabsf(theta) || m == D) break;
    }
    // q_{k+1}; warp 0 keeps the basis (read after the next step's first barrier)
    const float inv = 1.f / beta;
#pragma unroll
    for (int x = 0; x < VPL; ++x) q[x] = w[x] * inv;
    if (warp == 0) {
#pragma unroll
      for (int x = 0; x < VPL; ++x) basis[(k + 1) * D + VPL * lane + x] = q[x];
    }
  }
  if (tid == 0) mnorm[static_cast<size_t>(h) * nb + j] = sqrtf(fmaxf(theta, 0.f));
}

}  // namespace

int launch_block_heterogeneity(const void* k, const void* v, int in_bf16, int heads, int n,
                               int d, const float* kbar, const float* hbar, int spectral,
                               float* mnorm, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  const dim3 grid(nb, heads);
  auto run = [&](auto kern, const auto* kk, const auto* vv, size_t smem) -> int {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
    kern<<<grid, kThreads, smem, stream>>>(kk, vv, kbar, hbar, n, nb, mnorm);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  using BF = __nv_bfloat16;
  const BF* kb = static_cast<const BF*>(k);
  const BF* vb = static_cast<const BF*>(v);
  const float* kf = static_cast<const float*>(k);
  const float* vf = static_cast<const float*>(v);
  if (d == 128) {
    const size_t sm = HeteroSmem<128>::bytes(spectral != 0);
    if (in_bf16)
      return spectral ? run(hetero_kernel<BF, 128, true>, kb, vb, sm)
                      : run(hetero_kernel<BF, 128, false>, kb, vb, sm);
    return spectral ? run(hetero_kernel<float, 128, true>, kf, vf, sm)
                    : run(hetero_kernel<float, 128, false>, kf, vf, sm);
  }
  const size_t sm = HeteroSmem<64>::bytes(spectral != 0);
  if (in_bf16)
    return spectral ? run(hetero_kernel<BF, 64, true>, kb, vb, sm)
                    : run(hetero_kernel<BF, 64, false>, kb, vb, sm);
  return spectral ? run(hetero_kernel<float, 64, true>, kf, vf, sm)
                  : run(hetero_kernel<float, 64, false>, kf, vf, sm);
}

}  // namespace pisa
