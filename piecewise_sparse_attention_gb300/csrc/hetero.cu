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
// Frobenius norm of bf16 inputs with d = 128: frobenius_tc_kernel, a
// persistent CTA per SM streaming blocks through the tensor cores. Spectral
// norm of bf16 inputs with d = 128: spectral_tc_kernel, one CTA of four warps
// per (block, head), A and C = A^T A on the tensor cores and the Lanczos
// iteration on C held in registers, one row a thread. Every other case
// (float32 inputs, d = 64), one CTA (256 threads) per (block, head):
//   1-2. A = Kc^T V - Hbar into one 8x8 (d = 128) or 4x4 (d = 64) register
//      tile per thread, from the block's centred keys and values staged in
//      shared memory as float32; Frobenius: sum of squares, reduced in
//      double, done;
//   3. spectral: M_j^2 = lambda_max(A^T A) by the Lanczos iteration on
//      A^T A applied as A^T (A q) to the register tiles (A^T A is never
//      formed; one barrier per step).
// Both spectral kernels start from a dense vector plus A's largest row, stop
// on the residual of the top Ritz pair (relative 1e-6, below the float32
// error of forming A; at most d steps) and find the top Ritz value of the
// tridiagonal by Sturm-count multisection on each warp. Everything is float32
// except the Frobenius reduction. The Ritz values are lower bounds of
// lambda_max that converge to it; on the Wan-like blocks the stop comes after
// 10 to 16 steps.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "rowops.cuh"
#include "tc_ptx.cuh"

namespace pisa {
namespace {

constexpr int kThreads = 256;

template <int D>
struct HeteroSmem {
  static constexpr int KV = 2 * kBlock * D;        // centred keys, values (floats)
  // Lanczos buffers from float offset KV: per-warp partials [2][8][D], per-warp
  // alpha, beta, beta^2 [8][3][D]
  static constexpr int VEC = (2 * 8 + 8 * 3) * D;
  __host__ __device__ static constexpr size_t bytes(bool spectral) {
    return 1024 + (spectral ? static_cast<size_t>(KV + VEC) * 4 : static_cast<size_t>(KV) * 4);
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

// Sum of v over the 16 lanes of each half-warp, result in every lane:
// reduce-scatter (each round keeps the half of the values that the lane's bit
// selects and adds the partner's copy of it) down to one value a lane, plain
// sums over the remaining bits, then an all-gather by lane.
template <int TL>
__device__ __forceinline__ void halfwarp_allreduce(float (&v)[TL], int lane) {
  float h[TL];
#pragma unroll
  for (int i = 0; i < TL; ++i) h[i] = v[i];
#pragma unroll
  for (int r = 0; (TL >> r) > 1; ++r) {
    const int cnt = TL >> r, o = 8 >> r;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? h[i] : h[cnt / 2 + i];
      const float keep = upper ? h[cnt / 2 + i] : h[i];
      h[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float x = h[0];
#pragma unroll
  for (int o = 8 / TL; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
#pragma unroll
  for (int t = 0; t < TL; ++t) v[t] = __shfl_sync(0xffffffffu, x, (lane & 16) | (t * (16 / TL)));
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Stop test of the Lanczos iteration after m steps, run by a whole warp (every
// warp that calls it computes the same): theta, the largest eigenvalue of the
// tridiagonal T_m (diagonal wal, off-diagonal wbe, its squares wb2), and
// whether the iteration stops (residual of theta's Ritz pair below
// 1e-6 theta, a zero beta, or mmax steps).
__device__ __forceinline__ bool lanczos_check(const float* wal, const float* wbe, const float* wb2,
                                              int m, int mmax, float beta, int lane,
                                              float& theta) {
  // theta = largest eigenvalue of T_m, bracketed between the previous
  // checkpoint's theta (a lower bound: the top Ritz value only grows with
  // m) and the Gershgorin bound G. Sturm counts (eigenvalues below mu =
  // negative pivots of T_m - mu I) at 32 points a round: first a
  // geometric ladder lo + (G - lo) 2^(l - 31), which pins a theta that
  // moved little in one round, then even splits into 33.
  const float theta_prev = theta;
  float lo = theta, hi = 0.f;
  for (int i = lane; i < m; i += 32) {
    const float r = (i > 0 ? wbe[i - 1] : 0.f) + (i < m - 1 ? wbe[i] : 0.f);
    hi = fmaxf(hi, wal[i] + r);
  }
  hi = warp_max(hi);
  hi = hi * 1.000001f;
  lo = fminf(lo, hi);
  const float tiny = fmaxf(1e-30f * hi, 1e-36f);
  // lambda_max(T_m) < mu exactly when every leading principal minor of
  // mu I - T_m is positive (Sturm: the sign changes of the sequence count
  // the eigenvalues above mu). The minors follow the three-term recurrence
  // p_i = (mu - alpha_i) p_{i-1} - beta_{i-1}^2 p_{i-2}; scaled by 1 / G
  // a step grows them by at most the golden ratio, and every 16 steps
  // they are brought back by a power of two (no effect on the signs).
  // One fused multiply-add per step is on the dependent chain.
  const float ih = 1.f / hi, ih2 = ih * ih;
  auto all_below = [&](float mu) {
    const float mus = mu * ih;
    float p0 = 1.f, p1 = fmaf(-wal[0], ih, mus);
    bool pos = p1 > 0.f;
    auto step = [&](int i, float ai, float bi) {
      const float t = bi * ih2 * p0;
      const float p2 = fmaf(fmaf(-ai, ih, mus), p1, -t);
      pos = pos && p2 > 0.f;
      p0 = p1;
      p1 = p2;
      if ((i & 15) == 15) {
        const float mag = fmaxf(fabsf(p0), fabsf(p1));
        const float f = mag > 0x1p60f ? 0x1p-60f : (mag < 0x1p-60f && mag > 0.f ? 0x1p60f : 1.f);
        p0 *= f;
        p1 *= f;
      }
    };
#pragma unroll 4
    for (int i = 1; i < m; ++i) step(i, wal[i], wb2[i - 1]);
    return pos;
  };
  // stop at a bracket of 2.5e-7 hi, about two float32 ulps (theta then
  // carries <= 1.3e-7 relative error), or when a round cannot narrow it
  for (int round = 0; round < 12 && hi - lo > 2.5e-7f * hi; ++round) {
    const float mu = (round == 0)
                         ? (lane == 31 ? hi : lo + ldexpf(hi - lo, lane - 31))
                         : lo + (hi - lo) * static_cast<float>(lane + 1) * (1.f / 33.f);
    const unsigned all = __ballot_sync(0xffffffffu, all_below(mu));
    const int f = all ? __ffs(all) - 1 : 32;
    const float new_hi = (f < 32) ? __shfl_sync(0xffffffffu, mu, f & 31) : hi;
    const float new_lo = (f > 0) ? __shfl_sync(0xffffffffu, mu, (f - 1) & 31) : lo;
    if (new_hi == hi && new_lo == lo) break;
    hi = new_hi;
    lo = new_lo;
  }
  theta = 0.5f * (lo + hi);
  // a theta that still moved by more than 1e-4 has not converged: the
  // residual test is skipped
  const bool settled = beta == 0.f || m == mmax || theta - theta_prev <= 1e-4f * theta;
  if (settled) {
    // last component y_{m-1} of the normalised eigenvector of T_m, from the
    // bottom up (the stable direction: a converging Ritz vector decays
    // towards the end of the basis): x_{m-1} = 1, |x_i| = |x_{i+1}| |e_{i+1}|
    // / beta_i with e the pivots of the trailing blocks of T_m - hi I
    float xc = 1.f, xs = 1.f, xl = 1.f, e = wal[m - 1] - hi;
    auto up = [&](int i, float ai, float bi) {
      const float be = wbe[i];
      xc = (be > 0.f) ? __fdividef(xc * fabsf(e), be) : 0.f;
      if (xc > 1e18f) {
        xc *= 1e-18f;
        xs *= 1e-36f;
        xl *= 1e-18f;
      }
      xs = fmaf(xc, xc, xs);
      if (fabsf(e) < tiny) e = -tiny;
      e = ai - hi - __fdividef(bi, e);
    };
    for (int i = m - 2; i >= 0; --i) up(i, wal[i], wb2[i]);
    const float resid = beta * xl * rsqrtf(xs);
    if (beta == 0.f || resid <= 1e-6f * fabsf(theta) || m == mmax) return true;
  }
  return false;
}

constexpr long long kWaitLimit = 2000000000LL;

// One 16-byte chunk of 8 bf16 keys minus their block means mk, split into
// three bf16 terms by truncation: c1 = t with the low 16 bits of its float32
// pattern cleared, r = t - c1 (exact: the cleared bits, at most 16
// significant), c2 = r with its low 16 bits cleared, c3 = r - c2 (exact, at
// most 8 significant bits, so already a bf16 value). c1 + c2 + c3 = t
// exactly, and the low halves of all three are zero, so a byte permute packs
// two of them into one bf16 pair; no float-to-bf16 conversion is needed.
__device__ __forceinline__ void split3(uint4 kraw, const float (&mk)[8], uint4& w1, uint4& w2,
                                       uint4& w3) {
  const uint32_t kw[4] = {kraw.x, kraw.y, kraw.z, kraw.w};
  uint32_t p1[4], p2[4], p3[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint32_t u1[2], u2[2], u3[2];
#pragma unroll
    for (int y = 0; y < 2; ++y) {
      const float kv = __uint_as_float(y ? (kw[x] & 0xffff0000u) : (kw[x] << 16));
      const float t = kv - mk[2 * x + y];
      u1[y] = __float_as_uint(t) & 0xffff0000u;
      const float r = t - __uint_as_float(u1[y]);
      u2[y] = __float_as_uint(r) & 0xffff0000u;
      u3[y] = __float_as_uint(r - __uint_as_float(u2[y]));
    }
    // low half: the high 16 bits of the even channel, high half: the odd one's
    p1[x] = __byte_perm(u1[0], u1[1], 0x7632);
    p2[x] = __byte_perm(u2[0], u2[1], 0x7632);
    p3[x] = __byte_perm(u3[0], u3[1], 0x7632);
  }
  w1 = make_uint4(p1[0], p1[1], p1[2], p1[3]);
  w2 = make_uint4(p2[0], p2[1], p2[2], p2[3]);
  w3 = make_uint4(p3[0], p3[1], p3[2], p3[3]);
}

template <typename T, int D, bool SPECTRAL>
__global__ void __launch_bounds__(kThreads)
hetero_kernel(const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ kbar,
              const float* __restrict__ hbar, int n, int nb, float* __restrict__ mnorm,
              int32_t* status) {
  using S = HeteroSmem<D>;
  constexpr int TL = D / 16;  // register tile edge
  extern __shared__ __align__(16) unsigned char raw[];
  // 1024-byte aligned base (the swizzled tensor-core tiles need it)
  unsigned char* base = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
  float* sm = reinterpret_cast<float*>(base);
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int ty = tid / 16, tx = tid % 16;
  float acc[TL][TL];

  {
    constexpr int CH = Chunk<T>::kElems;
    float* sK = sm;                // [64][D] centred keys
    float* sV = sm + kBlock * D;   // [64][D] values
    const int r0 = j * kBlock;
    const int nj = min(kBlock, n - r0);

    // ---- 1. centred keys and values of block j -------------------------------
    const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D;
    const size_t gbase = (static_cast<size_t>(h) * n + r0) * D;
    for (int e = tid; e < kBlock * (D / CH); e += kThreads) {
      const int row = e / (D / CH), c0 = (e % (D / CH)) * CH;
      float fk[CH], fv[CH];
      if (row < nj) {
        Chunk<T>::load(k + gbase + static_cast<size_t>(row) * D + c0, fk);
        Chunk<T>::load(v + gbase + static_cast<size_t>(row) * D + c0, fv);
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

    // ---- 2. A = Kc^T V - Hbar, rows ty*TL.., columns tx*TL.. of this thread ---
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
    if (SPECTRAL) __syncthreads();  // every read of sK / sV is done before the Lanczos buffers
  }

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
  // q_0 as below; step k: w = A^T (A q_k) - beta_{k-1} q_{k-1},
  // alpha_k = q_k.w, w -= alpha_k q_k, beta_k = |w|, q_{k+1} = w / beta_k
  // (the plain three-term recurrence: in floating point the top Ritz value
  // converges as in exact arithmetic until it has converged, and lost
  // orthogonality only adds copies of converged values afterwards). The Ritz
  // values of the tridiagonal T_m (diagonal alpha, off-diagonal beta) are
  // lower bounds of lambda_max(C) up to rounding; at the checkpoints the
  // largest one, theta, is located by Sturm-count multisection and the step
  // stops once the residual of its Ritz vector, beta_{m-1} |y_{m-1}| (y the
  // normalised eigenvector of T_m), is below 1e-6 theta, or at m = D. By the
  // residual bound theta then lies within 1e-6 theta of an eigenvalue of
  // A^T A, so M_j = sqrt(theta) carries at most 5e-7 relative error from the
  // stop: less than forming A in float32 leaves in it (sums of 64 products
  // and the difference with Hbar, about 1e-6 of max ||H_j||).
  constexpr int VPL = D / 32;                    // vector elements per lane: VPL*lane ..
  constexpr int NW = kThreads / 32;
  float* part = sm + S::KV;                      // [2][NW][D] per-warp partial A^T (A q)
  float* wal = part + 2 * NW * D + warp * 3 * D; // this warp's copy of alpha [D],
  float* wbe = wal + D;                          //   beta [D]
  float* wb2 = wbe + D;                          //   and beta^2 [D]
  const int c0 = tx * TL;

  float q[VPL], qp[VPL];  // this lane's elements of q_k, q_{k-1} (every warp holds all)
  {
    // q_0: the fixed dense vector plus the row of A with the largest norm,
    // each normalised. A row of A is the top right singular vector weighted
    // by that row's share of it, so a dominant row (an outlier key channel)
    // starts the iteration close to it; the dense part keeps a share of every
    // direction, so no invariant subspace can hide the top singular value.
    float* cand = part + NW * D + D;  // [16] (norm^2, row) of each half-warp's best row
    float* srow = part + NW * D;      // [D] the chosen row
    float rn[TL];
#pragma unroll
    for (int a = 0; a < TL; ++a) {
      float t = 0.f;
#pragma unroll
      for (int b = 0; b < TL; ++b) t = fmaf(acc[a][b], acc[a][b], t);
      rn[a] = t;
    }
    halfwarp_allreduce<TL>(rn, lane);
    float bv = rn[0];
    int ba = 0;
#pragma unroll
    for (int a = 1; a < TL; ++a)
      if (rn[a] > bv) {
        bv = rn[a];
        ba = a;
      }
    if (tx == 0) {
      cand[2 * ty] = bv;
      cand[2 * ty + 1] = __int_as_float(ty * TL + ba);
    }
    __syncthreads();
    float best = cand[0];
    int brow = __float_as_int(cand[1]);
    for (int g = 1; g < kThreads / 16; ++g)
      if (cand[2 * g] > best) {  // strict: the lowest row wins a tie
        best = cand[2 * g];
        brow = __float_as_int(cand[2 * g + 1]);
      }
    if (ty == brow / TL) {
      const int am = brow % TL;
#pragma unroll
      for (int b = 0; b < TL; ++b) {
        float v = acc[0][b];
#pragma unroll
        for (int a = 1; a < TL; ++a) v = (a == am) ? acc[a][b] : v;
        srow[tx * TL + b] = v;
      }
    }
    __syncthreads();
    const float rinv = best > 0.f ? rsqrtf(best) : 0.f;
    float ss = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      const uint32_t e = static_cast<uint32_t>(VPL * lane + x);
      const uint32_t hsh = (e + 1u) * 2654435761u;
      q[x] = 0.25f + static_cast<float>(hsh >> 8) * (1.f / 16777216.f);  // in [0.25, 1.25)
      q[x] = (hsh & 1u) ? -q[x] : q[x];
      ss = fmaf(q[x], q[x], ss);
      qp[x] = 0.f;
    }
    const float dinv = rsqrtf(warp_sum(ss));
    ss = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      q[x] = fmaf(srow[VPL * lane + x], rinv, q[x] * dinv);
      ss = fmaf(q[x], q[x], ss);
    }
    const float inv = rsqrtf(warp_sum(ss));
#pragma unroll
    for (int x = 0; x < VPL; ++x) q[x] *= inv;
  }
  float theta = 0.f, beta_prev = 0.f;
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
      u[a] = t;
    }
    halfwarp_allreduce<TL>(u, lane);
    // this thread's part of A^T u: its rows, its columns; the warp's two row
    // groups summed. Double-buffered: the barrier of step k + 1 separates the
    // reads of buffer k & 1 from its next writes at step k + 2.
    float* pk = part + (k & 1) * NW * D;
    float z[TL];
#pragma unroll
    for (int b = 0; b < TL; ++b) {
      float t = 0.f;
#pragma unroll
      for (int a = 0; a < TL; ++a) t = fmaf(acc[a][b], u[a], t);
      z[b] = t + __shfl_xor_sync(0xffffffffu, t, 16);
    }
    if (lane < 16) {
#pragma unroll
      for (int b = 0; b < TL; b += 4)
        *reinterpret_cast<float4*>(pk + warp * D + c0 + b) = make_float4(z[b], z[b + 1], z[b + 2], z[b + 3]);
    }
    __syncthreads();
    float w[VPL];
#pragma unroll
    for (int x = 0; x < VPL; ++x) w[x] = 0.f;
#pragma unroll
    for (int p = 0; p < NW; ++p) {
      const float* src = pk + p * D + VPL * lane;
      if constexpr (VPL == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        w[0] += t.x;
        w[1] += t.y;
        w[2] += t.z;
        w[3] += t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        w[0] += t.x;
        w[1] += t.y;
      }
    }
#pragma unroll
    for (int x = 0; x < VPL; ++x) w[x] = fmaf(-beta_prev, qp[x], w[x]);
    float aa = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) aa = fmaf(w[x], q[x], aa);
    const float alpha = warp_sum(aa);
    float ss = 0.f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      w[x] = fmaf(-alpha, q[x], w[x]);
      ss = fmaf(w[x], w[x], ss);
    }
    const float beta = sqrtf(warp_sum(ss));
    if (lane == 0) {
      wal[k] = alpha;
      wbe[k] = beta;
      wb2[k] = beta * beta;
    }
    __syncwarp();
    const int m = k + 1;
    // checkpoints: every 2 steps from 8 to 24, every 4 up to 48, then every 8
    const bool check = (m <= 24) ? (m >= 8 && m % 2 == 0) : (m <= 48 ? (m % 4 == 0) : (m % 8 == 0));
    if (beta == 0.f || check || m == D) {
      if (lanczos_check(wal, wbe, wb2, m, D, beta, lane, theta)) break;
    }
    const float inv = 1.f / beta;
#pragma unroll
    for (int x = 0; x < VPL; ++x) {
      qp[x] = q[x];
      q[x] = w[x] * inv;
    }
    beta_prev = beta;
  }
  if (tid == 0) mnorm[static_cast<size_t>(h) * nb + j] = sqrtf(fmaxf(theta, 0.f));
}

// ---- spectral norm of bf16 blocks with d = 128: C = A^T A on the tensor cores --
// One CTA of four warps per (block, head), three CTAs per SM (128 TMEM
// columns, 69 KB of shared memory, at most 168 registers a thread each):
//   1. A = Kc^T V into TMEM columns [0, 128): the centred keys
//      Kc = K - kbar_j are split exactly into three bf16 terms c1 + c2 + c3
//      (split3), so Kc^T V = sum_s c_s^T V is three MMAs with exact bf16
//      products and float32 accumulation, both operands MN-major in the
//      128-byte swizzle (row r of a panel at r * 128 bytes, its 16-byte
//      chunk c at position c ^ (r & 7));
//   2. thread t reads row t of A (key channel t) into registers and
//      subtracts Hbar; A' = A - Hbar is then split exactly into three bf16
//      terms a1 + a2 + a3 (split3f), 64 key channels at a time, as
//      [64 key channels][128 value channels] operand tiles;
//   3. C = A'^T A' into the same TMEM columns (A has been read out) from the
//      six products a_s^T a_u with s + u <= 4 (1-based; the three left out
//      are below 2^-24 of C), K = 64 for each half of the key channels,
//      float32 accumulation;
//   4. C (symmetric) stays in TMEM; thread t reads its row t each step: a
//      Lanczos step is one 128-term dot product against q (read from shared
//      memory, the same address in every lane), two block sums and one
//      barrier to publish the next vector. No cross-thread product.
// The recurrence, start vector and stop test are those of hetero_kernel.
constexpr int kSpecThreads = 128;

struct SpecSmem {
  static constexpr int PANEL = kBlock * 128;   // form A: [64 tokens][64 channels] bf16
  static constexpr int TILE = 2 * PANEL;       // [64 tokens][128 channels]
  static constexpr int PANEL2 = 64 * 128;      // C operands: [64 rows][64 channels] bf16
  static constexpr int TILE2 = 2 * PANEL2;     // [64 rows][128 channels]
  static constexpr int OPS = 4 * TILE;         // form-A tiles; the three C operand tiles alias them
  static constexpr int VEC = OPS;              // floats: q [2][128], row [128], sums [2][4],
                                               // alpha, beta, beta^2 [3][128]
  static constexpr int NVEC = 256 + 128 + 8 + 3 * 128;
  static constexpr int CTRL = VEC + NVEC * 4;  // mbarrier, TMEM slot
  static constexpr size_t bytes = 1024 + CTRL + 64;
};

// Eight float32 values split exactly into three bf16 terms by truncation (as
// split3 does for centred keys), packed into bf16 pairs.
__device__ __forceinline__ void split3f(const float* x, uint4& w1, uint4& w2, uint4& w3) {
  uint32_t p1[4], p2[4], p3[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t u1[2], u2[2], u3[2];
#pragma unroll
    for (int y = 0; y < 2; ++y) {
      const float t = x[2 * i + y];
      u1[y] = __float_as_uint(t) & 0xffff0000u;
      const float r = t - __uint_as_float(u1[y]);
      u2[y] = __float_as_uint(r) & 0xffff0000u;
      u3[y] = __float_as_uint(r - __uint_as_float(u2[y]));
    }
    p1[i] = __byte_perm(u1[0], u1[1], 0x7632);
    p2[i] = __byte_perm(u2[0], u2[1], 0x7632);
    p3[i] = __byte_perm(u3[0], u3[1], 0x7632);
  }
  w1 = make_uint4(p1[0], p1[1], p1[2], p1[3]);
  w2 = make_uint4(p2[0], p2[1], p2[2], p2[3]);
  w3 = make_uint4(p3[0], p3[1], p3[2], p3[3]);
}

// Sum over the CTA's 128 threads, the same value in every thread (fixed
// order); `slots` alternates between two sets of four, so a set is rewritten
// only after every thread has read it.
__device__ __forceinline__ float block_sum128(float x, float* slots, int& calls, int warp,
                                              int lane) {
  x = warp_sum(x);
  float* sl = slots + 4 * (calls & 1);
  ++calls;
  if (lane == 0) sl[warp] = x;
  __syncthreads();
  return (sl[0] + sl[1]) + (sl[2] + sl[3]);
}

__global__ void __launch_bounds__(kSpecThreads, 3)
spectral_tc_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                   const float* __restrict__ kbar, const float* __restrict__ hbar, int n, int nb,
                   float* __restrict__ mnorm, int32_t* status) {
  constexpr int D = 128;
  using S = SpecSmem;
  extern __shared__ __align__(16) unsigned char raw[];
  unsigned char* base = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
  float* vec = reinterpret_cast<float*>(base + S::VEC);
  float* qbuf = vec;              // [2][128]
  float* srow = vec + 256;        // [128]
  float* sums = vec + 384;        // [2][4]
  float* wal = vec + 392;         // [128] alpha, then beta, beta^2
  float* wbe = wal + D;
  float* wb2 = wbe + D;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + S::CTRL);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int r0 = j * kBlock, nj = min(kBlock, n - r0);
  const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;

  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 128);
    tc::tmem_relinquish();
  }
  // ---- 1. A = Kc^T V: split keys, copy values into the form-A tiles ----------
  {
    // chunk i of this thread: token tid / 16 + 8 i, channels 8 (tid % 16) ..;
    // every load is issued before any is used
    constexpr int PER = kBlock * (D / 8) / kSpecThreads;  // 8
    const int ch = tid % (D / 8);
    const size_t gbase = (static_cast<size_t>(h) * n + r0) * D + 8 * ch;
    const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D + 8 * ch;
    const float4 m0 = __ldg(reinterpret_cast<const float4*>(kb));
    const float4 m1 = __ldg(reinterpret_cast<const float4*>(kb) + 1);
    uint4 kr[PER], vr[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int r = tid / (D / 8) + 8 * i;
      kr[i] = vr[i] = make_uint4(0u, 0u, 0u, 0u);
      if (r < nj) {
        kr[i] = __ldg(reinterpret_cast<const uint4*>(k + gbase + static_cast<size_t>(r) * D));
        vr[i] = __ldg(reinterpret_cast<const uint4*>(v + gbase + static_cast<size_t>(r) * D));
      }
    }
    const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int r = tid / (D / 8) + 8 * i;
      const uint32_t off = (ch >> 3) * S::PANEL + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      uint4 w1 = make_uint4(0u, 0u, 0u, 0u), w2 = w1, w3 = w1;
      if (r < nj) split3(kr[i], mk, w1, w2, w3);
      *reinterpret_cast<uint4*>(base + 0 * S::TILE + off) = w1;
      *reinterpret_cast<uint4*>(base + 1 * S::TILE + off) = w2;
      *reinterpret_cast<uint4*>(base + 2 * S::TILE + off) = w3;
      *reinterpret_cast<uint4*>(base + 3 * S::TILE + off) = vr[i];
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  constexpr uint32_t IDESC = tc::idesc_bf16_f32(D, D, true) | (1u << 15);  // A, B MN-major
  const uint32_t b0 = tc::smem_u32(base);
  if (tid == 0) {
    const uint32_t va = b0 + 3 * S::TILE;
#pragma unroll
    for (int sp = 0; sp < 3; ++sp)
#pragma unroll
      for (int ks = 0; ks < kBlock / 16; ++ks)
        tc::mma_ss(tmem, tc::smem_desc_sw128(b0 + sp * S::TILE + ks * 2048, S::PANEL, 1024),
                   tc::smem_desc_sw128(va + ks * 2048, S::PANEL, 1024), IDESC,
                   (sp > 0 || ks > 0) ? 1u : 0u);
    tc::mma_commit(bar);
  }
  int zero = 0;
  bool ok = tc::mbar_wait(bar, 0, &zero, kWaitLimit);
  if (!ok) {
    if (tid == 0) report(status, PISA_ERR_TIMEOUT);
    tc::mbar_wait(bar, 0, &zero, kWaitLimit);  // the MMAs may still read the tiles
  }
  ok = __syncthreads_and(ok);
  tc::tc_fence_after();

  // ---- 2. A' = A - Hbar, row tid, into registers ----------------------------------
  const float* hrow = hbar + (static_cast<size_t>(h) * D + tid) * D;
  float a[D];
  float rn = 0.f;  // |row tid of A'|^2
  if (ok) {
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      uint32_t rr[32];
      tc::tmem_ld32(tmem + lane_off + 32 * q, rr);
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 hx = __ldg(reinterpret_cast<const float4*>(hrow + 32 * q) + e4);
        a[32 * q + 4 * e4 + 0] = -hx.x;
        a[32 * q + 4 * e4 + 1] = -hx.y;
        a[32 * q + 4 * e4 + 2] = -hx.z;
        a[32 * q + 4 * e4 + 3] = -hx.w;
      }
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        a[32 * q + e] += __uint_as_float(rr[e]);
        rn = fmaf(a[32 * q + e], a[32 * q + e], rn);
      }
    }
  }
  // the largest row of A' (lowest row on ties), kept for the start vector
  float best = rn;
  int brow = tid;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int orow = __shfl_xor_sync(0xffffffffu, brow, o);
    if (ob > best || (ob == best && orow < brow)) {
      best = ob;
      brow = orow;
    }
  }
  if (lane == 0) {
    sums[2 * warp] = best;
    sums[2 * warp + 1] = __int_as_float(brow);
  }
  tc::tc_fence_before();
  __syncthreads();  // every read of A is done: its TMEM columns take C
  tc::tc_fence_after();
  best = sums[0];
  brow = __float_as_int(sums[1]);
  for (int w = 1; w < 4; ++w)
    if (sums[2 * w] > best) {  // strict: the lowest row wins a tie
      best = sums[2 * w];
      brow = __float_as_int(sums[2 * w + 1]);
    }
  if (tid == brow) {
#pragma unroll
    for (int e4 = 0; e4 < D / 4; ++e4)
      *reinterpret_cast<float4*>(srow + 4 * e4) =
          make_float4(a[4 * e4], a[4 * e4 + 1], a[4 * e4 + 2], a[4 * e4 + 3]);
  }
  // ---- 3. C = A'^T A', the key channels in two halves of 64 ----------------------
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    if (ok && warp / 2 == half) {
      const int row = tid - 64 * half;  // row of the half's operand tiles
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {  // 16-byte chunk of 8 value channels
        const uint32_t off = (ch >> 3) * S::PANEL2 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
        uint4 w1, w2, w3;
        split3f(a + 8 * ch, w1, w2, w3);
        *reinterpret_cast<uint4*>(base + 0 * S::TILE2 + off) = w1;
        *reinterpret_cast<uint4*>(base + 1 * S::TILE2 + off) = w2;
        *reinterpret_cast<uint4*>(base + 2 * S::TILE2 + off) = w3;
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (ok && tid == 0) {
      constexpr int PS[6] = {0, 0, 1, 0, 2, 1}, PU[6] = {0, 1, 0, 2, 0, 1};
#pragma unroll
      for (int p = 0; p < 6; ++p)
#pragma unroll
        for (int ks = 0; ks < kBlock / 16; ++ks)
          tc::mma_ss(tmem,
                     tc::smem_desc_sw128(b0 + PS[p] * S::TILE2 + ks * 2048, S::PANEL2, 1024),
                     tc::smem_desc_sw128(b0 + PU[p] * S::TILE2 + ks * 2048, S::PANEL2, 1024),
                     IDESC, (half > 0 || p > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(bar);
    }
    // commits 2 and 3 of the barrier complete its phases 1 and 2
    if (ok) {
      ok = tc::mbar_wait(bar, (half + 1) & 1, &zero, kWaitLimit);
      if (!ok) {
        if (tid == 0) report(status, PISA_ERR_TIMEOUT);
        tc::mbar_wait(bar, (half + 1) & 1, &zero, kWaitLimit);  // the MMAs may still read
      }
    }
    ok = __syncthreads_and(ok);
    tc::tc_fence_after();
  }
  int calls = 0;
  float qv, qp = 0.f;  // this thread's entries of q_k, q_{k-1}
  {
    const uint32_t hsh = (static_cast<uint32_t>(tid) + 1u) * 2654435761u;
    float dq = 0.25f + static_cast<float>(hsh >> 8) * (1.f / 16777216.f);  // in [0.25, 1.25)
    dq = (hsh & 1u) ? -dq : dq;
    const float dinv = rsqrtf(block_sum128(dq * dq, sums, calls, warp, lane));
    const float rinv = best > 0.f ? rsqrtf(best) : 0.f;
    qv = fmaf(srow[tid], rinv, dq * dinv);
    qv *= rsqrtf(block_sum128(qv * qv, sums, calls, warp, lane));
  }
  qbuf[tid] = qv;
  __syncthreads();
  float theta = 0.f, beta_prev = 0.f;
  for (int kk = 0; ok && kk < D; ++kk) {
    // u = C q, this thread's entry: row tid of C (TMEM lane tid, read 64
    // columns at a time) against the whole of q
    const float4* qc = reinterpret_cast<const float4*>(qbuf + (kk & 1) * D);
    float u[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hc = 0; hc < D / 64; ++hc) {
      uint32_t c0[32], c1[32];
      tc::tmem_ld32(tmem + lane_off + 64 * hc, c0);
      tc::tmem_ld32(tmem + lane_off + 64 * hc + 32, c1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 x = qc[16 * hc + i];
        const uint32_t(&cc)[32] = i < 8 ? c0 : c1;
        const int b = 4 * (i & 7), o = 4 * (i & 1);
        u[o + 0] = fmaf(__uint_as_float(cc[b + 0]), x.x, u[o + 0]);
        u[o + 1] = fmaf(__uint_as_float(cc[b + 1]), x.y, u[o + 1]);
        u[o + 2] = fmaf(__uint_as_float(cc[b + 2]), x.z, u[o + 2]);
        u[o + 3] = fmaf(__uint_as_float(cc[b + 3]), x.w, u[o + 3]);
      }
    }
    float w = fmaf(-beta_prev, qp, ((u[0] + u[1]) + (u[2] + u[3])) + ((u[4] + u[5]) + (u[6] + u[7])));
    const float alpha = block_sum128(w * qv, sums, calls, warp, lane);
    w = fmaf(-alpha, qv, w);
    const float beta = sqrtf(block_sum128(w * w, sums, calls, warp, lane));
    if (tid == 0) {
      wal[kk] = alpha;
      wbe[kk] = beta;
      wb2[kk] = beta * beta;
    }
    // the next vector, published with the step's alpha and beta
    const float qn = w * (1.f / beta);
    qbuf[((kk + 1) & 1) * D + tid] = qn;
    __syncthreads();
    const int m = kk + 1;
    // checkpoints: every 2 steps from 8 to 24, every 4 up to 48, then every 8
    const bool check = (m <= 24) ? (m >= 8 && m % 2 == 0) : (m <= 48 ? (m % 4 == 0) : (m % 8 == 0));
    if (beta == 0.f || check || m == D) {
      if (lanczos_check(wal, wbe, wb2, m, D, beta, lane, theta)) break;
    }
    qp = qv;
    qv = qn;
    beta_prev = beta;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {  // every TMEM read is done
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
  if (ok && tid == 0) mnorm[static_cast<size_t>(h) * nb + j] = sqrtf(fmaxf(theta, 0.f));
}

// ---- H_j itself for pisa_block_stats (bf16, d = 128) ------------------------------
// H_j = Kc^T V formed exactly as step 1 of spectral_tc_kernel (three MMAs over
// the exact bf16 split of the centred keys, float32 accumulation), then
// thread t reads row t (key channel t) from TMEM into a padded staging area
// and the CTA writes the 128 x 128 result out in coalesced 16-byte pieces,
// as float32 or rounded to bf16. One CTA of four warps per (block, head).
struct BlockHSmem {
  static constexpr int STG_LD = 128 + 4;              // staging row stride (floats)
  static constexpr int STG = 128 * STG_LD * 4;        // 67.6 KB, over the form-A tiles
  static constexpr int CTRL = STG;                    // mbarrier, TMEM slot
  static constexpr size_t bytes = 1024 + CTRL + 64;
  static_assert(STG >= SpecSmem::OPS, "the staging area covers the form-A tiles");
};

__global__ void __launch_bounds__(kSpecThreads, 3)
block_h_tc_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                  const float* __restrict__ kbar, int n, int nb, void* __restrict__ hmat,
                  int h_bf16, int32_t* status) {
  constexpr int D = 128;
  using S = SpecSmem;
  extern __shared__ __align__(16) unsigned char raw[];
  unsigned char* base = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + BlockHSmem::CTRL);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid / 32;
  const int r0 = j * kBlock, nj = min(kBlock, n - r0);
  const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;

  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 128);
    tc::tmem_relinquish();
  }
  {
    // chunk i of this thread: token tid / 16 + 8 i, channels 8 (tid % 16) ..;
    // every load is issued before any is used
    constexpr int PER = kBlock * (D / 8) / kSpecThreads;  // 8
    const int ch = tid % (D / 8);
    const size_t gbase = (static_cast<size_t>(h) * n + r0) * D + 8 * ch;
    const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D + 8 * ch;
    const float4 m0 = __ldg(reinterpret_cast<const float4*>(kb));
    const float4 m1 = __ldg(reinterpret_cast<const float4*>(kb) + 1);
    uint4 kr[PER], vr[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int r = tid / (D / 8) + 8 * i;
      kr[i] = vr[i] = make_uint4(0u, 0u, 0u, 0u);
      if (r < nj) {
        kr[i] = __ldg(reinterpret_cast<const uint4*>(k + gbase + static_cast<size_t>(r) * D));
        vr[i] = __ldg(reinterpret_cast<const uint4*>(v + gbase + static_cast<size_t>(r) * D));
      }
    }
    const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int r = tid / (D / 8) + 8 * i;
      const uint32_t off = (ch >> 3) * S::PANEL + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      uint4 w1 = make_uint4(0u, 0u, 0u, 0u), w2 = w1, w3 = w1;
      if (r < nj) split3(kr[i], mk, w1, w2, w3);
      *reinterpret_cast<uint4*>(base + 0 * S::TILE + off) = w1;
      *reinterpret_cast<uint4*>(base + 1 * S::TILE + off) = w2;
      *reinterpret_cast<uint4*>(base + 2 * S::TILE + off) = w3;
      *reinterpret_cast<uint4*>(base + 3 * S::TILE + off) = vr[i];
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    constexpr uint32_t IDESC = tc::idesc_bf16_f32(D, D, true) | (1u << 15);  // A, B MN-major
    const uint32_t b0 = tc::smem_u32(base);
    const uint32_t va = b0 + 3 * S::TILE;
#pragma unroll
    for (int sp = 0; sp < 3; ++sp)
#pragma unroll
      for (int ks = 0; ks < kBlock / 16; ++ks)
        tc::mma_ss(tmem, tc::smem_desc_sw128(b0 + sp * S::TILE + ks * 2048, S::PANEL, 1024),
                   tc::smem_desc_sw128(va + ks * 2048, S::PANEL, 1024), IDESC,
                   (sp > 0 || ks > 0) ? 1u : 0u);
    tc::mma_commit(bar);
  }
  int zero = 0;
  bool ok = tc::mbar_wait(bar, 0, &zero, kWaitLimit);
  if (!ok) {
    if (tid == 0) report(status, PISA_ERR_TIMEOUT);
    tc::mbar_wait(bar, 0, &zero, kWaitLimit);  // the MMAs may still read the tiles
  }
  ok = __syncthreads_and(ok);
  tc::tc_fence_after();
  // row tid of H_j into the staging area (stride 132 floats: conflict-free
  // 16-byte stores across the warp's rows)
  float* stg = reinterpret_cast<float*>(base);
  if (ok) {
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      uint32_t rr[32];
      tc::tmem_ld32(tmem + lane_off + 32 * q, rr);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4)
        *reinterpret_cast<float4*>(stg + tid * BlockHSmem::STG_LD + 32 * q + 4 * e4) =
            make_float4(__uint_as_float(rr[4 * e4]), __uint_as_float(rr[4 * e4 + 1]),
                        __uint_as_float(rr[4 * e4 + 2]), __uint_as_float(rr[4 * e4 + 3]));
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
  if (!ok) return;  // CTA-uniform
  // coalesced write-out: 16-byte piece e of the block's D x D values
  const size_t hbase = (static_cast<size_t>(h) * nb + j) * D * D;
  if (h_bf16) {
    uint2* dst = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(hmat) + hbase);
    for (int e = tid; e < D * D / 4; e += kSpecThreads) {
      const int row = e / (D / 4), c4 = e % (D / 4);
      const float4 x = *reinterpret_cast<const float4*>(stg + row * BlockHSmem::STG_LD + 4 * c4);
      dst[e] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    }
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(hmat) + hbase);
    for (int e = tid; e < D * D / 4; e += kSpecThreads) {
      const int row = e / (D / 4), c4 = e % (D / 4);
      dst[e] = *reinterpret_cast<const float4*>(stg + row * BlockHSmem::STG_LD + 4 * c4);
    }
  }
}

// ---- Frobenius norm streamed through the tensor cores (bf16, d = 128) -------
// M_j = ||H_j - Hbar||_F needs no register tile of A, so this path streams:
// one persistent CTA per SM walks a contiguous range of (head, block) items
// with three warp roles that hand items to each other through mbarriers
// (no CTA-wide barrier inside the loop):
//   - the issuer (one thread) starts the bulk copies of an item's 64 key rows,
//     64 value rows (16 KB each, contiguous in [heads, n, d]) and kbar row
//     into stage t % 3 of a ring, three items ahead; when the split warps
//     have filled tile set t % 2 and the epilogue has released accumulator
//     t % 2, it issues the 12 MMAs of H_j and commits them to done[t % 2];
//   - 8 split warps wait for the copies and for the MMAs of item t - 2 (the
//     tile set is then free), split the centred keys into c1, c2, c3 (split3)
//     and copy V into tile set t % 2 (the swizzled layout of the spectral kernel's form-A tiles);
//   - 8 epilogue warps wait for done, read the accumulator (warp w: TMEM lanes
//     32 (w % 4) .., the key channels; 64 value channels) and Hbar, which they
//     keep in TMEM columns 256-383 while the head stays the same, release the
//     accumulator and sum squares in float32 (64 per thread, a butterfly over
//     the warp, the 8 warps in order after a named barrier: deterministic,
//     relative error a few 1e-6 on M_j^2).
// A wait that runs out sets a shared abort flag that ends every role's loop;
// the issuer then waits (bounded) for its copies and MMAs still in flight.
constexpr int kFrobSplitWarps = 8;
constexpr int kFrobEpiWarps = 8;
constexpr int kFrobThreads = 32 * (kFrobSplitWarps + kFrobEpiWarps + 1);
constexpr int kFrobStages = 3;

struct FrobSmem {
  static constexpr int D = 128;
  static constexpr int PANEL = kBlock * 128;     // [64 tokens][64 channels] bf16
  static constexpr int TILE = 2 * PANEL;         // [64 tokens][128 channels]
  static constexpr int SET = 4 * TILE;           // c1, c2, c3, V
  static constexpr int RAW = kBlock * D * 2;     // one block's rows of K (or V)
  static constexpr int STAGE = 2 * RAW + D * 4;  // K rows, V rows, kbar row
  static constexpr int RING = 2 * SET;           // byte offsets from the 1024-aligned base
  // full[3], done[2], ready[2], tfree[2] mbarriers, the TMEM slot, the abort flag
  static constexpr int CTRL = RING + kFrobStages * STAGE;
  static constexpr int PART = CTRL + 128;  // [2][8] per-warp sums
  static constexpr size_t bytes = 1024 + PART + 2 * kFrobEpiWarps * sizeof(float);
};
static_assert(FrobSmem::bytes <= 232448, "one CTA's opt-in shared memory");
static_assert(FrobSmem::STAGE % 16 == 0 && FrobSmem::RAW % 16 == 0, "bulk copy alignment");
static_assert(kBlock * (FrobSmem::D / 8) == 4 * 32 * kFrobSplitWarps, "four chunks a thread");

// OR of `pred` over the `nthreads` threads (whole warps) that meet at named
// barrier `id`; every one of them gets the result.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kFrobThreads, 1)
frobenius_tc_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const float* __restrict__ kbar, const float* __restrict__ hbar, int n, int nb,
                    int items, float* __restrict__ mnorm, int32_t* status) {
  using S = FrobSmem;
  constexpr int D = S::D;
  extern __shared__ __align__(16) unsigned char raw[];
  unsigned char* base = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + S::CTRL);
  uint64_t* done = full + kFrobStages;  // MMAs of item t complete (count 1: the commit)
  uint64_t* ready = done + 2;           // tile set written (count: the split warps)
  uint64_t* tfree = ready + 2;          // accumulator read (count: the epilogue warps)
  uint32_t* slot = reinterpret_cast<uint32_t*>(tfree + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  float* part = reinterpret_cast<float*>(base + S::PART);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int first = static_cast<int>(static_cast<long long>(blockIdx.x) * items / gridDim.x);
  const int cnt =
      static_cast<int>(static_cast<long long>(blockIdx.x + 1) * items / gridDim.x) - first;

  if (tid == 0) {
    for (int s = 0; s < kFrobStages; ++s) tc::mbar_init(full + s, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(done + b, 1);
      tc::mbar_init(ready + b, kFrobSplitWarps);
      tc::mbar_init(tfree + b, kFrobEpiWarps);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(slot, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *slot;
  int loads = 0, mmas = 0;  // the issuer's counts of started copies and MMA groups

  if (warp < kFrobSplitWarps) {
    // ---- split warps: stage t % 3 -> tile set t % 2 ----
    const int ch = tid % 16;  // 16-byte chunk of 8 channels, the same for all four rows
    for (int t = 0; t < cnt; ++t) {
      const int stage = t % kFrobStages;
      const int j = (first + t) % nb, nj = min(kBlock, n - j * kBlock);
      bool got = tc::mbar_wait(full + stage, (t / kFrobStages) & 1, abort_flag, kWaitLimit);
      if (got && t >= 2)
        got = tc::mbar_wait(done + (t & 1), ((t - 2) >> 1) & 1, abort_flag, kWaitLimit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const unsigned char* st = base + S::RING + stage * S::STAGE;
      unsigned char* set = base + (t & 1) * S::SET;
      const float4 m0 = *reinterpret_cast<const float4*>(st + 2 * S::RAW + 32 * ch);
      const float4 m1 = *reinterpret_cast<const float4*>(st + 2 * S::RAW + 32 * ch + 16);
      const float mk[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = tid / 16 + 16 * i;
        const uint32_t off = (ch >> 3) * S::PANEL + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        uint4 w1 = make_uint4(0u, 0u, 0u, 0u), w2 = w1, w3 = w1, vr = w1;
        if (r < nj) {
          const uint4 kr = *reinterpret_cast<const uint4*>(st + r * 256 + 16 * ch);
          vr = *reinterpret_cast<const uint4*>(st + S::RAW + r * 256 + 16 * ch);
          split3(kr, mk, w1, w2, w3);
        }
        *reinterpret_cast<uint4*>(set + 0 * S::TILE + off) = w1;
        *reinterpret_cast<uint4*>(set + 1 * S::TILE + off) = w2;
        *reinterpret_cast<uint4*>(set + 2 * S::TILE + off) = w3;
        *reinterpret_cast<uint4*>(set + 3 * S::TILE + off) = vr;
      }
      tc::fence_proxy_async_smem();  // the tiles, visible to the MMAs
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(ready + (t & 1));
    }
  } else if (warp < kFrobSplitWarps + kFrobEpiWarps) {
    // ---- epilogue warps: accumulator t % 2 minus Hbar, sum of squares ----
    const int ew = warp - kFrobSplitWarps;
    const int c = 32 * (warp & 3) + lane, cseg = 64 * (ew >> 2);
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t hcol = tmem + lane_base + 256 + cseg;
    int hcached = -1;
    for (int u = 0; u < cnt; ++u) {
      const int h = (first + u) / nb;
      if (h != hcached) {  // this warp's part of Hbar into its TMEM columns
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          const float4* hb = reinterpret_cast<const float4*>(
              hbar + (static_cast<size_t>(h) * D + c) * D + cseg + 32 * q);
          uint32_t hh[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = __ldg(hb + e);
            hh[4 * e] = __float_as_uint(x.x);
            hh[4 * e + 1] = __float_as_uint(x.y);
            hh[4 * e + 2] = __float_as_uint(x.z);
            hh[4 * e + 3] = __float_as_uint(x.w);
          }
          tc::tmem_st32(hcol + 32 * q, hh);
        }
        tc::tmem_wait_st();
        hcached = h;
      }
      const bool got = __all_sync(
          0xffffffffu, tc::mbar_wait(done + (u & 1), (u >> 1) & 1, abort_flag, kWaitLimit));
      if (got) {
        tc::tc_fence_after();
        const uint32_t acc = tmem + lane_base + (u & 1) * 128 + cseg;
        float sq = 0.f;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          uint32_t rr[32], hh[32];
          tc::tmem_ld32(acc + 32 * q, rr);
          tc::tmem_ld32(hcol + 32 * q, hh);
          tc::tmem_wait_ld();
          if (q == 1) {  // the accumulator is read: the MMAs of item u + 2 may use it
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tfree + (u & 1));
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(rr[e]) - __uint_as_float(hh[e]);
            sq = fmaf(x, x, sq);
          }
        }
        const float w = warp_sum(sq);
        if (lane == 0) part[(u & 1) * kFrobEpiWarps + ew] = w;
      } else if (lane == 0) {
        *abort_flag = 1;
      }
      // every epilogue warp meets here once per item and all take the same
      // decision, so none is left waiting at the named barrier
      if (bar_red_or(1, 32 * kFrobEpiWarps, !got || *abort_flag != 0)) break;
      if (ew == 0 && lane == 0) {
        float t2 = 0.f;
        for (int w = 0; w < kFrobEpiWarps; ++w) t2 += part[(u & 1) * kFrobEpiWarps + w];
        mnorm[first + u] = sqrtf(t2);
      }
    }
  } else if (lane == 0) {
    // ---- issuer: copies three items ahead, the MMAs of item t ----
    auto issue_load = [&](int u) {
      const int it = first + u, h = it / nb, j = it - h * nb, r0 = j * kBlock;
      const uint32_t rows = static_cast<uint32_t>(min(kBlock, n - r0)) * D * 2;
      unsigned char* st = base + S::RING + (u % kFrobStages) * S::STAGE;
      uint64_t* bar = full + u % kFrobStages;
      const size_t g = (static_cast<size_t>(h) * n + r0) * D;
      tc::mbar_arrive_expect_tx(bar, 2 * rows + D * 4);
      tc::bulk_load(st, k + g, rows, bar);
      tc::bulk_load(st + S::RAW, v + g, rows, bar);
      tc::bulk_load(st + 2 * S::RAW, kbar + (static_cast<size_t>(h) * nb + j) * D, D * 4, bar);
    };
    for (; loads < min(cnt, kFrobStages); ++loads) issue_load(loads);
    constexpr uint32_t IDESC = tc::idesc_bf16_f32(D, D, true) | (1u << 15);  // A, B MN-major
    // descriptors of the two tile sets, built once: an MMA adds its offset / 16
    const uint64_t dset0 = tc::smem_desc_sw128(tc::smem_u32(base), S::PANEL, 1024);
    const uint64_t dset1 = tc::smem_desc_sw128(tc::smem_u32(base + S::SET), S::PANEL, 1024);
    for (int t = 0; t < cnt; ++t) {
      bool got = tc::mbar_wait(ready + (t & 1), (t >> 1) & 1, abort_flag, kWaitLimit);
      if (got && t >= 2)
        got = tc::mbar_wait(tfree + (t & 1), ((t - 2) >> 1) & 1, abort_flag, kWaitLimit);
      if (!got) {
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const uint64_t dset = (t & 1) ? dset1 : dset0;
      const uint32_t acc = tmem + (t & 1) * 128;
#pragma unroll
      for (int sp = 0; sp < 3; ++sp)
#pragma unroll
        for (int ks = 0; ks < kBlock / 16; ++ks)
          tc::mma_ss(acc, dset + ((sp * S::TILE + ks * 2048) >> 4),
                     dset + ((3 * S::TILE + ks * 2048) >> 4), IDESC, (sp > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(done + (t & 1));
      ++mmas;
      // ready[t % 2] means the split warps have read stage t % 3
      if (t + kFrobStages < cnt) issue_load(loads++);
    }
  }
  __syncthreads();  // every role has left its loop; the abort flag is final
  if (tid == kFrobThreads - 32 && *abort_flag != 0) {
    // the copies and MMAs that may still be in flight: the last three copies
    // and the last two MMA groups started (each wait bounded)
    report(status, PISA_ERR_TIMEOUT);
    int zero = 0;
    for (int u = max(0, loads - kFrobStages); u < loads; ++u)
      tc::mbar_wait(full + u % kFrobStages, (u / kFrobStages) & 1, &zero, kWaitLimit);
    for (int u = max(0, mmas - 2); u < mmas; ++u)
      tc::mbar_wait(done + (u & 1), (u >> 1) & 1, &zero, kWaitLimit);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_block_h_tc(const void* k, const void* v, int heads, int n, const float* kbar,
                      void* hmat, int h_bf16, int32_t* status, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  PISA_CUDA_TRY(cudaFuncSetAttribute(block_h_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(BlockHSmem::bytes)));
  block_h_tc_kernel<<<dim3(nb, heads), kSpecThreads, BlockHSmem::bytes, stream>>>(
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), kbar, n, nb, hmat,
      h_bf16, status);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

int launch_block_heterogeneity(const void* k, const void* v, int in_bf16, int heads, int n,
                               int d, const float* kbar, const float* hbar, int spectral,
                               float* mnorm, int32_t* status, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  const dim3 grid(nb, heads);
  auto run = [&](auto kern, const auto* kk, const auto* vv, size_t smem) -> int {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
    kern<<<grid, kThreads, smem, stream>>>(kk, vv, kbar, hbar, n, nb, mnorm, status);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  using BF = __nv_bfloat16;
  const BF* kb = static_cast<const BF*>(k);
  const BF* vb = static_cast<const BF*>(v);
  const float* kf = static_cast<const float*>(k);
  const float* vf = static_cast<const float*>(v);
  if (d == 128 && in_bf16 && !spectral) {  // streamed Frobenius norm
    int dev = 0, sms = 0;
    PISA_CUDA_TRY(cudaGetDevice(&dev));
    PISA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int items = heads * nb;
    PISA_CUDA_TRY(cudaFuncSetAttribute(frobenius_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(FrobSmem::bytes)));
    frobenius_tc_kernel<<<min(items, sms), kFrobThreads, FrobSmem::bytes, stream>>>(
        kb, vb, kbar, hbar, n, nb, items, mnorm, status);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  }
  if (d == 128) {
    const size_t sm = HeteroSmem<128>::bytes(spectral != 0);
    if (in_bf16) {  // spectral, A and C = A^T A on the tensor cores
      PISA_CUDA_TRY(cudaFuncSetAttribute(spectral_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SpecSmem::bytes)));
      spectral_tc_kernel<<<grid, kSpecThreads, SpecSmem::bytes, stream>>>(kb, vb, kbar, hbar, n,
                                                                          nb, mnorm, status);
      PISA_CHECK_LAUNCH();
      return PISA_OK;
    }
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
