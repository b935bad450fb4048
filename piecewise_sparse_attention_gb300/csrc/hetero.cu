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
//   3. spectral: C = A^T A (symmetric, positive semidefinite) held in registers
//      (each thread its 8x8 / 4x4 tile), Householder reduction of C to a
//      tridiagonal T (same eigenvalues) with the reflector and C' v exchanged
//      through shared memory, and the largest eigenvalue of T by Sturm-count
//      multisection on one warp (32 trial points per round);
//      M_j = sqrt(lambda_max).
// Everything is float32 except the Frobenius reduction; the tridiagonal
// reduction is backward stable, so lambda_max carries a relative error of a
// few units in the last place of C.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

constexpr int kThreads = 256;

template <int D>
struct HeteroSmem {
  static constexpr int LD = D + 1;  // padded row stride of A and C
  static constexpr int KV = 2 * kBlock * D;
  static constexpr int MAT = D * LD;
  static constexpr int BIG = KV > MAT ? KV : MAT;
  static constexpr int VEC = BIG;  // v [2][D], p [2][D], v.p parts [2][16], diagonal, off-diagonal
  static constexpr size_t bytes(bool spectral) {
    return spectral ? (static_cast<size_t>(BIG) + 6 * D + 32) * 4 + 64
                    : static_cast<size_t>(KV) * 4 + 64;
  }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
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
  constexpr int LD = S::LD;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm;                // [64][D] centred keys
  float* sV = sm + kBlock * D;   // [64][D] values
  float* sA = sm;                // [D][LD]: A, then C (after the K/V phase)
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

  // ---- 3. spectral norm: C = A^T A, tridiagonalise, largest eigenvalue ----------
  __syncthreads();  // every read of sK / sV is done before A overwrites them
#pragma unroll
  for (int a = 0; a < TL; ++a)
#pragma unroll
    for (int b = 0; b < TL; ++b) sA[(ty * TL + a) * LD + tx * TL + b] = acc[a][b];
  __syncthreads();
  // C = A^T A stays in registers: this thread owns rows tr0.., columns c0..
  const int tr0 = ty * TL, c0 = tx * TL;
  float c[TL][TL];
#pragma unroll
  for (int a = 0; a < TL; ++a)
#pragma unroll
    for (int b = 0; b < TL; ++b) c[a][b] = 0.f;
#pragma unroll 4
  for (int i = 0; i < D; ++i) {
    float x[TL], y[TL];
#pragma unroll
    for (int a = 0; a < TL; ++a) {
      x[a] = sA[i * LD + tr0 + a];
      y[a] = sA[i * LD + c0 + a];
    }
#pragma unroll
    for (int a = 0; a < TL; ++a)
#pragma unroll
      for (int b = 0; b < TL; ++b) c[a][b] = fmaf(x[a], y[b], c[a][b]);
  }
  float* vbuf = sm + S::VEC;  // Householder vector v (unit length), [2][D]
  float* pbuf = vbuf + 2 * D; // p = C' v, [2][D]
  float* kbuf = pbuf + 2 * D; // per row group partial v.p, [2][16]
  float* dg = kbuf + 32;      // diagonal of T
  float* e2 = dg + D;         // squared off-diagonal of T
  const unsigned half = 0xffffu << (16 * (ty & 1));  // the 16 lanes sharing this row group

  // Householder step kk maps column kk below the diagonal onto its first
  // entry; the trailing block C' becomes (I - 2vv^T) C' (I - 2vv^T) =
  // C' - v w^T - w v^T, w = 2 (p - (v.p) v), p = C' v. Vectors alternate
  // between two buffers, so one barrier after the reflector and one after p
  // suffice per step.
  for (int kk = 0; kk < D - 2; ++kk) {
    float* hv = vbuf + (kk & 1) * D;
    float* hp = pbuf + (kk & 1) * D;
    float* kp = kbuf + (kk & 1) * 16;
    if (ty == kk / TL) {
      // the 16 lanes holding row kk (= column kk) build the reflector
      const int rr = kk - tr0;
      float row[TL], x[TL];
#pragma unroll
      for (int e = 0; e < TL; ++e) {
        float val = 0.f;
#pragma unroll
        for (int a = 0; a < TL; ++a) val = (a == rr) ? c[a][e] : val;
        row[e] = val;
        x[e] = (c0 + e > kk) ? val : 0.f;
      }
      float ss = 0.f, x0 = 0.f, dd = 0.f;
#pragma unroll
      for (int e = 0; e < TL; ++e) {
        ss = fmaf(x[e], x[e], ss);
        x0 += (c0 + e == kk + 1) ? x[e] : 0.f;
        dd += (c0 + e == kk) ? row[e] : 0.f;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(half, ss, o);
        x0 += __shfl_xor_sync(half, x0, o);
        dd += __shfl_xor_sync(half, dd, o);
      }
      const float sigma = sqrtf(ss);
      const float alpha = (x0 > 0.f) ? -sigma : sigma;
      const float vn2 = 2.f * (ss + fabsf(x0) * sigma);  // |x - alpha e1|^2
      const float inv = (vn2 > 0.f) ? rsqrtf(vn2) : 0.f;
#pragma unroll
      for (int e = 0; e < TL; ++e) hv[c0 + e] = ((c0 + e == kk + 1) ? x[e] - alpha : x[e]) * inv;
      if (tx == 0) {
        dg[kk] = dd;
        e2[kk] = alpha * alpha;
      }
    }
    __syncthreads();
    float vr[TL], vc[TL], p[TL];
#pragma unroll
    for (int a = 0; a < TL; ++a) {
      vr[a] = hv[tr0 + a];
      vc[a] = hv[c0 + a];
      p[a] = 0.f;
    }
    if (__any_sync(0xffffffffu, tr0 + TL - 1 > kk)) {  // this warp holds trailing rows
#pragma unroll
      for (int a = 0; a < TL; ++a) {
        float s = 0.f;
#pragma unroll
        for (int b = 0; b < TL; ++b) s = fmaf(c[a][b], vc[b], s);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        p[a] = (tr0 + a > kk) ? s : 0.f;
      }
    }
    float kpart = 0.f;
#pragma unroll
    for (int a = 0; a < TL; ++a) kpart = fmaf(vr[a], p[a], kpart);
    if (tx == 0) kp[ty] = kpart;
#pragma unroll
    for (int a = 0; a < TL; ++a)
      if (tx == a) hp[tr0 + a] = p[a];
    __syncthreads();
    if (tr0 + TL - 1 > kk) {
      float K = 0.f;
#pragma unroll
      for (int t = 0; t < 16; ++t) K += kp[t];
      float wr[TL], wc[TL];
#pragma unroll
      for (int a = 0; a < TL; ++a) {
        wr[a] = 2.f * fmaf(-K, vr[a], p[a]);
        wc[a] = 2.f * fmaf(-K, vc[a], hp[c0 + a]);
      }
#pragma unroll
      for (int a = 0; a < TL; ++a)
#pragma unroll
        for (int b = 0; b < TL; ++b) c[a][b] -= fmaf(vr[a], wc[b], wr[a] * vc[b]);
    }
  }
  if (ty == 15 && tx == 15) {  // the final 2 x 2 block
    dg[D - 2] = c[TL - 2][TL - 2];
    dg[D - 1] = c[TL - 1][TL - 1];
    e2[D - 2] = c[TL - 2][TL - 1] * c[TL - 2][TL - 1];
  }
  __syncthreads();

  // largest eigenvalue of T: Sturm counts (number of eigenvalues below mu =
  // number of negative pivots of the LDL^T factorisation of T - mu I) at 32
  // points per round inside a Gershgorin interval
  if (warp == 0) {
    float lo = 0.f, hi = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float r = sqrtf(i > 0 ? e2[i - 1] : 0.f) + sqrtf(i < D - 1 ? e2[i] : 0.f);
      hi = fmaxf(hi, dg[i] + r);
      lo = fminf(lo, dg[i] - r);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    }
    hi *= 1.0001f;
    const float tiny = 1e-30f;
    for (int round = 0; round < 8 && hi - lo > 1e-7f * fabsf(hi); ++round) {
      const float mu = lo + (hi - lo) * static_cast<float>(lane + 1) * (1.f / 33.f);
      int below = 0;
      float q = dg[0] - mu;
      below += q < 0.f;
      for (int i = 1; i < D; ++i) {
        if (fabsf(q) < tiny) q = -tiny;
        q = dg[i] - mu - e2[i - 1] / q;
        below += q < 0.f;
      }
      const unsigned all = __ballot_sync(0xffffffffu, below == D);  // lambda_max < mu
      const int f = all ? __ffs(all) - 1 : 32;
      const float new_hi = (f < 32) ? __shfl_sync(0xffffffffu, mu, f & 31) : hi;
      const float new_lo = (f > 0) ? __shfl_sync(0xffffffffu, mu, (f - 1) & 31) : lo;
      hi = new_hi;
      lo = new_lo;
    }
    if (lane == 0)
      mnorm[static_cast<size_t>(h) * nb + j] = sqrtf(fmaxf(0.5f * (lo + hi), 0.f));
  }
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
