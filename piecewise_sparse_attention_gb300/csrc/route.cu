// Block routing: S_i = band(i) U top-k{ j outside the band } by the pooled
// score s * qbar_i . kbar_j, lower block index first among equal scores.
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Figure 4 "Prepare Phase" and Algorithm 1 step 2; the band as
// in the Piecewise-Taylor-Attention README ("Knobs", band=b).
//
// Since s > 0 the ranking is that of x_ij = qbar_i . kbar_j. The selection is
// the one defined by the exact value of x_ij for the given float32 inputs,
// obtained in two stages:
//
//   1. every score is computed in float32 (x~) with the a-priori error bound
//      |x~ - x| <= E_i = gamma_d ||qbar_i|| max_j ||kbar_j|| (gamma_d = d u / (1 - d u),
//      u = 2^-24, Cauchy-Schwarz on sum |q_c k_c|, 2% margin);
//   2. a bracket t_lo <= t_hi of the k-th largest x~ with #(x~ > t_hi) <= k <=
//      #(x~ >= t_lo), found by bisection on the score value with warp-wide
//      counts (it usually ends on a t with exactly k scores >= t, then
//      t_lo = t_hi = t). Every candidate with x~ > t_hi + 2E_i is certainly
//      selected (fewer than k others can reach its exact score), every one
//      with x~ < t_lo - 2E_i certainly not (k others are certainly above it),
//      and only the few in between are decided exactly: when they are all in
//      or all out nothing more is computed, else each gets an exact
//      double-float score (error-free products and sums, ~2^-44 relative) and
//      the exact selection with the lowest-index tie-break is made among them.
//
// If that ambiguous set is larger than a per-warp buffer (mass near-ties),
// the exact selection among it recomputes the double-float scores on each
// pass of a 64-bit radix select instead of storing them.
//
// Covariance-aware variant (Section 3.3 Eq. 11): the ranking key becomes
// y_ij = s x_ij + b_j with b_j = log(M_j + eps) evaluated in double and held
// as a float pair (hi + lo). Stage 1 uses y~ = fl(s x~ + b_hi) with the bound
// s E_i + u (s |x~| + 2 max|b|) (one rounding, the lo part dropped); stage 2
// forms s x + b_hi + b_lo from the double-float dot product with error-free
// products and sums. An optional per-pair bonus (the second-order ranking
// bonus of the Piecewise-Taylor-Attention README) is added the same way: one
// more rounding in stage 1, an error-free sum in stage 2.
//
// A CTA owns R query blocks of one head (32, 16 or 8, as many as 64 KB of
// score rows hold). Phase A is a register-tiled float32 product: the key
// blocks are staged in shared memory in chunks (64 KB: 256 keys x 64 channels,
// 512 x 32 or 1024 x 16, double-buffered with coalesced cp.async copies and an
// XOR swizzle that makes the per-key reads conflict-free), and each thread
// accumulates 8 query rows x 4 key blocks, one sequential FMA chain over the
// channels per score (the chain the stage-1 bound assumes). The scores go to
// shared memory as order-preserving 32-bit keys. Phase B: each warp takes one
// row at a time, brackets the threshold, decides the ambiguous candidates and
// emits the set in ascending order with ballots.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr size_t kScoreBudget = 65536;  // bytes of shared memory for a CTA's score rows
constexpr int kAmbCap = 128;            // exact keys a warp can hold for one row
constexpr int kChunkFloats = 8192;      // one staged key chunk: 32 KB

// 16-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Position of 16-byte column c4 of staged key row kk (rows of F columns):
// eight consecutive rows read at the same c4 land in eight different 16-byte
// bank groups.
template <int F>
__device__ __forceinline__ int swz(int kk, int c4) {
  if constexpr (F >= 8) return kk * F + (c4 ^ (kk & 7));
  else return kk * F + (c4 ^ ((kk / (8 / F)) & (F - 1)));
}

__device__ __forceinline__ float ord32_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Warp-wide radix select over items [0, m): K* = the take-th largest key among
// the valid items (`src(i, key)` returns false for an excluded item), and
// *eq_take = how many items equal to K* belong to the top `take` (the lowest
// item indices among them). BITS = key width (32 or 64).
template <int BITS, typename Src>
__device__ uint64_t warp_radix_select(int m, int take, Src src, uint32_t* hist, int lane,
                                      int* eq_take) {
  uint64_t prefix = 0, pmask = 0;
  int need = take;
  for (int shift = BITS - 8; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0u;
    __syncwarp();
    for (int i0 = 0; i0 < m; i0 += 32) {
      const int i = i0 + lane;
      uint64_t key = 0;
      const bool valid = i < m && src(i, key);
      const bool match = valid && ((key & pmask) == prefix);
      const int dg = match ? static_cast<int>((key >> shift) & 0xffu) : -1;
      if (__ballot_sync(0xffffffffu, match)) {
        const unsigned peers = __match_any_sync(0xffffffffu, dg);
        if (match && (__ffs(peers) - 1) == lane) atomicAdd(&hist[dg], __popc(peers));
      }
    }
    __syncwarp();
    // digit holding the need-th largest key: bins scanned 255..0
    uint32_t cnt8[8];
    uint32_t mine = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      cnt8[t] = hist[255 - (lane * 8 + t)];
      mine += cnt8[t];
    }
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - mine;
    int found = -1, above = 0;
    if (excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need)) {
      uint32_t run = excl;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (found < 0) {
          if (run + cnt8[t] >= static_cast<uint32_t>(need)) {
            found = 255 - (lane * 8 + t);
            above = static_cast<int>(run);
          } else {
            run += cnt8[t];
          }
        }
      }
    }
    const int src_lane = __ffs(__ballot_sync(0xffffffffu, found >= 0)) - 1;
    found = __shfl_sync(0xffffffffu, found, src_lane);
    above = __shfl_sync(0xffffffffu, above, src_lane);
    prefix |= static_cast<uint64_t>(found) << shift;
    pmask |= 0xffull << shift;
    need -= above;
    __syncwarp();
  }
  *eq_take = need;
  return prefix;
}

// b = log(m + eps) in double as hi + lo; a value that is not a norm
// (negative, NaN, inf) is taken as 0 (the caller reports it)
__device__ __forceinline__ void bias_pair(float m, float eps, float& hi, float& lo) {
  if (!(m >= 0.f && m <= 3.4e38f)) m = 0.f;
  const double b = log(static_cast<double>(m) + static_cast<double>(eps));
  hi = static_cast<float>(b);
  lo = static_cast<float>(b - static_cast<double>(hi));
}

// key of s (hi + lo) + (b_hi + b_lo) + beta in double-float
__device__ __forceinline__ uint64_t biased_key(float hi, float lo, float s, float b_hi,
                                               float b_lo, float beta) {
  const float p = __fmul_rn(s, hi);
  const float pe = __fmaf_rn(s, hi, -p);  // exact error of s * hi
  float S, E, S2, E2;
  two_sum(p, b_hi, S, E);
  two_sum(S, beta, S2, E2);
  E = __fadd_rn(__fadd_rn(E, E2), __fadd_rn(__fadd_rn(pe, __fmul_rn(s, lo)), b_lo));
  float rh, rl;
  fast_two_sum(S2, E, rh, rl);
  return dfloat_key(rh, rl);
}

template <int D, bool BIAS>
__device__ __forceinline__ uint64_t score_key(const float* __restrict__ q,
                                              const float* __restrict__ k, float s, float m,
                                              float eps, bool has_m, float beta) {
  DFloat acc;
  const float4* k4 = reinterpret_cast<const float4*>(k);
#pragma unroll 4
  for (int c4 = 0; c4 < D / 4; ++c4) {
    const float4 kv = __ldg(k4 + c4);
    const float4 qv = *reinterpret_cast<const float4*>(q + 4 * c4);
    acc.fma_acc(qv.x, kv.x);
    acc.fma_acc(qv.y, kv.y);
    acc.fma_acc(qv.z, kv.z);
    acc.fma_acc(qv.w, kv.w);
  }
  if (!BIAS) return dfloat_key(acc.hi, acc.lo);
  float b_hi = 0.f, b_lo = 0.f;
  if (has_m) bias_pair(m, eps, b_hi, b_lo);
  return biased_key(acc.hi, acc.lo, s, b_hi, b_lo, beta);
}

// score_key with the channels split over the warp: each lane accumulates its
// D / 32 channels in double-float, then a butterfly merges the lanes' pairs.
// The merge is commutative (TwoSum's error term is exact either way round),
// so every lane ends with the same key. For a few candidates this is much
// shorter than one lane walking all D channels.
template <int D, bool BIAS>
__device__ __forceinline__ uint64_t score_key_warp(const float* __restrict__ q,
                                                   const float* __restrict__ k, float s, float m,
                                                   float eps, bool has_m, float beta, int lane) {
  constexpr int PER = D / 32;
  DFloat acc;
#pragma unroll
  for (int c = 0; c < PER; ++c) acc.fma_acc(q[PER * lane + c], __ldg(k + PER * lane + c));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, acc.hi, off);
    const float olo = __shfl_xor_sync(0xffffffffu, acc.lo, off);
    acc.merge(ohi, olo);
  }
  if (!BIAS) return dfloat_key(acc.hi, acc.lo);
  float b_hi = 0.f, b_lo = 0.f;
  if (has_m) bias_pair(m, eps, b_hi, b_lo);
  return biased_key(acc.hi, acc.lo, s, b_hi, b_lo, beta);
}

// Warp-wide count of the row's keys >= tk (non-candidates hold the sentinel
// 0, which is below every score's key); the row is padded to a multiple of 4.
__device__ __forceinline__ int count_ge(const uint32_t* __restrict__ kr, int nbp, uint32_t tk,
                                        int lane) {
  int c = 0;
  for (int j = 4 * lane; j < nbp; j += 128) {
    const uint4 k4 = *reinterpret_cast<const uint4*>(kr + j);
    c += (k4.x >= tk) + (k4.y >= tk) + (k4.z >= tk) + (k4.w >= tk);
  }
  return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
}

// RL: the CTA's row layout (32, 16 or 8 rows: RL / 8 groups of 8 rows, the
// warps of one row group splitting the keys of a chunk); R <= RL rows are live.
// Two CTAs share an SM (at most ~112 KB of shared memory each), so one CTA's
// selection phase overlaps the other's products.
template <int D, bool BIAS, int RL>
__global__ void __launch_bounds__(kThreads, BIAS ? 1 : 2)
route_kernel(const float* __restrict__ qbar, const float* __restrict__ kbar, int nb, int R,
             int topk, int band, int32_t* __restrict__ idx, int32_t* __restrict__ cnt,
             int max_sel, const float* __restrict__ mnorm, float eps, float scale,
             int32_t* status, int n_sink, const float* __restrict__ bonus) {
  constexpr int NKB = 1;
  constexpr int RW = RL / 8;            // row groups
  constexpr int KW = kWarps / RW;       // warps per row group (key groups)
  constexpr int KT = RL == 8 ? 2 : 4;   // key blocks per thread
  constexpr int CK = KW * 32 * KT;      // key blocks per chunk
  constexpr int CH = kChunkFloats / CK; // channels per chunk
  constexpr int F = CH / 4;             // 16-byte columns per staged row
  constexpr int NPASS = D / CH;         // channel slices per key chunk
  static_assert(D % CH == 0 && (F == 2 || F == 4 || F % 8 == 0), "chunk shape");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int nbp = (nb + 3) & ~3;  // score row stride (16-byte rows)
  const int nwords = ceil_div(nb, 32);
  float* qs = reinterpret_cast<float*>(smem_raw);                        // [RL][D]
  float* kb = qs + RL * D;                                                // [NKB][chunk]
  uint32_t* keys = reinterpret_cast<uint32_t*>(kb + NKB * kChunkFloats); // [R][nbp]
  uint32_t* selw = keys + static_cast<size_t>(R) * nbp;                   // [warp][nwords]
  float* bhi = reinterpret_cast<float*>(selw + kWarps * nwords);          // [nb] (BIAS)
  // phase B's other per-warp buffers reuse the staged key chunk
  uint64_t* akey = reinterpret_cast<uint64_t*>(kb);                        // [warp][cap]
  int32_t* aidx = reinterpret_cast<int32_t*>(akey + kWarps * kAmbCap);   // [warp][cap]
  uint32_t* hist = reinterpret_cast<uint32_t*>(aidx + kWarps * kAmbCap); // [warp][256]
  static_assert(kWarps * kAmbCap * 12 + kWarps * 256 * 4 <= NKB * kChunkFloats * 4, "phase B");
  __shared__ uint32_t s_kn2max;  // max ||kbar_j||^2 as float bits (non-negative)
  __shared__ uint32_t s_bmax;    // max |b_j| as float bits

  const int h = blockIdx.y;
  const int i0 = blockIdx.x * R;
  const int rows = min(R, nb - i0);
  const int tid = threadIdx.x;
  const float* qh = qbar + static_cast<size_t>(h) * nb * D;
  const float* kh = kbar + static_cast<size_t>(h) * nb * D;
  const float* mh = (BIAS && mnorm) ? mnorm + static_cast<size_t>(h) * nb : nullptr;
  // per-pair bonus rows of this head (BIAS, optional)
  const float* bon = (BIAS && bonus) ? bonus + static_cast<size_t>(h) * nb * nb : nullptr;

  if (tid == 0) {
    s_kn2max = 0u;
    s_bmax = 0u;
  }
  for (int e = tid; e < RL * D; e += kThreads)
    qs[e] = e < rows * D ? qh[static_cast<size_t>(i0) * D + e] : 0.f;
  // padding keys of every row: the sentinel 0 counts as no candidate
  for (int e = tid; e < rows * (nbp - nb); e += kThreads)
    keys[(e / (nbp - nb)) * nbp + nb + e % (nbp - nb)] = 0u;
  __syncthreads();
  if (BIAS) {
    // b_j = log(M_j + eps) in double, split into two floats
    float bm = 0.f;
    for (int j = tid; j < nb; j += kThreads) {
      if (mh) {
        const float m = mh[j];
        if (!(m >= 0.f && m <= 3.4e38f)) report(status, PISA_ERR_DEVICE_CHECK);  // not a norm
        float lo;
        bias_pair(m, eps, bhi[j], lo);
      } else {
        bhi[j] = 0.f;
      }
      bm = fmaxf(bm, fabsf(bhi[j]));
    }
    atomicMax(&s_bmax, __float_as_uint(bm));
    __syncthreads();
  }

  // ---- phase A: float32 scores x~ and the largest key norm -----------------
  // Steps walk the key chunks, each in NPASS channel slices; the copy of the
  // next step is in flight while the current one is computed (NKB = 2).
  const int warp = tid / 32, lane = tid % 32;
  const int rg = warp % RW, kg = warp / RW;
  const int nsteps = ceil_div(nb, CK) * NPASS;
  auto issue = [&](int step) {
    const int j0 = (step / NPASS) * CK, cs = (step % NPASS) * CH;
    float* dst = kb + (NKB == 2 ? (step & 1) : 0) * kChunkFloats;
    // rows past the last key block are not copied (a key group that starts
    // past it skips its products; the tail of a started group is read but its
    // scores are never stored)
    const int rows_in = min(CK, nb - j0);
    for (int e = tid; e < rows_in * F; e += kThreads) {
      const int kk = e / F, c4 = e % F;
      cp_async16(dst + 4 * swz<F>(kk, c4), kh + static_cast<size_t>(j0 + kk) * D + cs + 4 * c4, 16);
    }
    cp_async_commit();
  };
  float kn2max = 0.f;
  float acc[8][KT];
  float kn[CK / kThreads];
  issue(0);
  for (int step = 0; step < nsteps; ++step) {
    const int pass = step % NPASS, j0 = (step / NPASS) * CK;
    if (NKB == 2 && step + 1 < nsteps) {
      issue(step + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* kc = kb + (NKB == 2 ? (step & 1) : 0) * kChunkFloats;
    if (pass == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < KT; ++m) acc[i][m] = 0.f;
#pragma unroll
      for (int a = 0; a < CK / kThreads; ++a) kn[a] = 0.f;
    }
    // key norms: thread tid owns keys tid, tid + 256, ... of the chunk
#pragma unroll
    for (int a = 0; a < CK / kThreads; ++a) {
      const int kk = tid + a * kThreads;
      if (j0 + kk >= nb) continue;
#pragma unroll 4
      for (int c4 = 0; c4 < F; ++c4) {
        const float4 v = *reinterpret_cast<const float4*>(kc + 4 * swz<F>(kk, c4));
        kn[a] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, kn[a]))));
      }
    }
    // scores: rows rg*8 .. rg*8+7, key blocks kg*32*KT + lane + 32 m of the chunk
    const float* qr = qs + rg * 8 * D + pass * CH;
    const bool live = j0 + kg * 32 * KT < nb;  // warp-uniform
#pragma unroll 2
    for (int c4 = 0; c4 < (live ? F : 0); ++c4) {
      float4 qv[8], kv[KT];
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = *reinterpret_cast<const float4*>(qr + i * D + 4 * c4);
#pragma unroll
      for (int m = 0; m < KT; ++m)
        kv[m] = *reinterpret_cast<const float4*>(kc + 4 * swz<F>(kg * 32 * KT + lane + 32 * m, c4));
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int m = 0; m < KT; ++m) {
          acc[i][m] = fmaf(qv[i].x, kv[m].x, acc[i][m]);
          acc[i][m] = fmaf(qv[i].y, kv[m].y, acc[i][m]);
          acc[i][m] = fmaf(qv[i].z, kv[m].z, acc[i][m]);
          acc[i][m] = fmaf(qv[i].w, kv[m].w, acc[i][m]);
        }
    }
    if (pass == NPASS - 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        if (r < rows) {
#pragma unroll
          for (int m = 0; m < KT; ++m) {
            const int j = j0 + kg * 32 * KT + lane + 32 * m;
            if (j < nb)
              keys[static_cast<size_t>(r) * nbp + j] = ord32(
                  BIAS ? fmaf(scale, acc[i][m], bhi[j]) +
                             (bon ? bon[static_cast<size_t>(i0 + r) * nb + j] : 0.f)
                       : acc[i][m]);
          }
        }
      }
#pragma unroll
      for (int a = 0; a < CK / kThreads; ++a)
        if (j0 + tid + a * kThreads < nb) kn2max = fmaxf(kn2max, kn[a]);
    }
    __syncthreads();  // the buffer just read is the next copy's destination
    if (NKB == 1 && step + 1 < nsteps) issue(step + 1);
  }
  atomicMax(&s_kn2max, __float_as_uint(kn2max));
  __syncthreads();
  // the norm itself is computed in float32: a relative slack of 1e-4 covers it
  const float kn_max = sqrtf(__uint_as_float(s_kn2max));

  // ---- phase B: per-row selection, one warp per row at a time --------------
  constexpr float kU = 5.9604645e-8f;  // 2^-24
  constexpr float kGamma = (D * kU) / (1.f - D * kU);
  uint64_t* ak = akey + warp * kAmbCap;
  int32_t* ai = aidx + warp * kAmbCap;
  uint32_t* hr = hist + warp * 256;
  uint32_t* sr = selw + warp * nwords;
  for (int r = warp; r < rows; r += kWarps) {
    const int i = i0 + r;
    const float* qrow = qs + r * D;
    uint32_t* kr = keys + static_cast<size_t>(r) * nbp;
    // forced blocks: the band and the first n_sink blocks
    const int lo_band = max(0, i - band), hi_band = min(nb - 1, i + band);
    const int n_forced = (hi_band - lo_band + 1) + n_sink -
                         max(0, min(hi_band, n_sink - 1) - lo_band + 1);
    const int n_cand = nb - n_forced;
    const int take = min(topk, n_cand);
    auto is_cand = [&](int j) { return (j < lo_band || j > hi_band) && j >= n_sink; };
    // exact double-float key of candidate j
    auto exact_key = [&](int j) {
      return score_key<D, BIAS>(qrow, kh + static_cast<size_t>(j) * D, scale,
                                mh ? mh[j] : 0.f, eps, mh != nullptr,
                                bon ? bon[static_cast<size_t>(i) * nb + j] : 0.f);
    };

    for (int w = lane; w < nwords; w += 32) sr[w] = 0u;
    __syncwarp();

    if (take == n_cand) {
      // every candidate is selected: the whole row
      for (int w = lane; w < nwords; w += 32) {
        const int valid = min(32, nb - w * 32);
        sr[w] = (valid == 32) ? 0xffffffffu : ((1u << valid) - 1u);
      }
    } else if (take > 0) {
      // the forced blocks leave the count: sentinel keys
      for (int j = lo_band + lane; j <= hi_band; j += 32) kr[j] = 0u;
      for (int j = lane; j < n_sink; j += 32) kr[j] = 0u;
      // error bound of this row's float32 scores (doubled: both ends of a gap)
      float qn2 = 0.f;
      for (int c = lane; c < D; c += 32) qn2 = fmaf(qrow[c], qrow[c], qn2);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) qn2 += __shfl_xor_sync(0xffffffffu, qn2, o);
      const float qk = sqrtf(qn2) * kn_max;
      float e2 = 2.f * 1.02f * kGamma * qk * 1.0001f + 1e-30f;
      float betamax = 0.f;  // largest |bonus| of this row
      if (BIAS && bon) {
        for (int j = lane; j < nb; j += 32) betamax = fmaxf(betamax, fabsf(bon[static_cast<size_t>(i) * nb + j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) betamax = fmaxf(betamax, __shfl_xor_sync(0xffffffffu, betamax, o));
      }
      if (BIAS)  // s E_i, the roundings of s x~ + b_hi and of + bonus, the dropped b_lo
        e2 = 2.f * 1.02f * (scale * 0.5f * e2 +
                            kU * (2.f * scale * qk * 1.01f + 3.f * __uint_as_float(s_bmax) + betamax)) +
             1e-30f;
      __syncwarp();

      // bracket [t_lo, t_hi] of the take-th largest x~: start from the
      // candidates' range and narrow it on the value until exactly `take` keys
      // are >= the probe or the bracket is narrower than the error window
      // rows of up to 512 blocks are searched from registers (16 keys a
      // lane), longer ones from shared memory
      const bool in_regs = nbp <= 512;
      uint4 rk[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int jj = 4 * lane + 128 * a;
        rk[a] = (in_regs && jj < nbp) ? *reinterpret_cast<const uint4*>(kr + jj)
                                      : make_uint4(0u, 0u, 0u, 0u);
      }
      auto count_from = [&](uint32_t tk) -> int {
        if (!in_regs) return count_ge(kr, nbp, tk, lane);
        int c = 0;
#pragma unroll
        for (int a = 0; a < 4; ++a)
          c += (rk[a].x >= tk) + (rk[a].y >= tk) + (rk[a].z >= tk) + (rk[a].w >= tk);
        return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
      };
      uint32_t kmax = 0u, kmin = 0xffffffffu;
      auto fold = [&](uint32_t key) {
        if (key != 0u) {
          kmax = max(kmax, key);
          kmin = min(kmin, key);
        }
      };
      if (in_regs) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          fold(rk[a].x);
          fold(rk[a].y);
          fold(rk[a].z);
          fold(rk[a].w);
        }
      } else {
        for (int j = lane; j < nb; j += 32) fold(kr[j]);
      }
      kmax = __reduce_max_sync(0xffffffffu, kmax);
      kmin = __reduce_min_sync(0xffffffffu, kmin);
      // The next probe interpolates the count linearly between the bracket's
      // ends (c_lo = #(x~ >= t_lo), c_hi ~ #(x~ >= t_hi)), kept within the
      // middle three quarters of the bracket so that it always shrinks.
      float t_lo = ord32_inv(kmin), t_hi = ord32_inv(kmax);
      float c_lo = static_cast<float>(n_cand), c_hi = 1.f;
      for (int it = 0; it < 64 && t_hi - t_lo > e2; ++it) {
        float f = (c_lo - (static_cast<float>(take) + 0.5f)) / fmaxf(c_lo - c_hi, 1.f);
        f = fminf(fmaxf(f, 0.125f), 0.875f);
        float mid = t_lo + f * (t_hi - t_lo);
        if (!(mid > t_lo && mid < t_hi)) mid = t_lo + 0.5f * (t_hi - t_lo);
        if (!(mid > t_lo && mid < t_hi)) break;  // no representable point inside
        const int c = count_from(ord32(mid));
        if (c == take) {
          t_lo = t_hi = mid;
          break;
        }
        if (c > take) {
          t_lo = mid;
          c_lo = static_cast<float>(c);
        } else {
          t_hi = mid;
          c_hi = static_cast<float>(c);
        }
      }
      const float hi_v = t_hi + e2, lo_v = t_lo - e2;

      // certain picks (x~ > t_hi + 2E) and the ambiguous set (in between)
      int n_def = 0, n_amb = 0;
      if (in_regs) {
        // from the register window: lane L holds keys 4 L + 128 a + c, which
        // are bits 4 (L % 8) + c of bitmask word 4 a + L / 8; the 8 lanes of
        // a word OR their nibbles together (forced blocks and padding hold
        // the sentinel 0, which no score maps to)
        uint32_t* amw = hr;  // ambiguous-bit words (the histogram is idle here)
        int dcnt = 0, acnt = 0;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const uint32_t kk[4] = {rk[a].x, rk[a].y, rk[a].z, rk[a].w};
          uint32_t dn = 0u, an = 0u;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const bool cand = kk[c] != 0u;
            const float xv = ord32_inv(kk[c]);
            const bool def = cand && xv > hi_v;
            const bool amb = cand && !def && xv >= lo_v;
            dn |= static_cast<uint32_t>(def) << c;
            an |= static_cast<uint32_t>(amb) << c;
          }
          dcnt += __popc(dn);
          acnt += __popc(an);
          uint32_t dw = dn << (4 * (lane & 7)), aw = an << (4 * (lane & 7));
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            dw |= __shfl_xor_sync(0xffffffffu, dw, o);
            aw |= __shfl_xor_sync(0xffffffffu, aw, o);
          }
          const int w = 4 * a + (lane >> 3);
          if ((lane & 7) == 0 && w < nwords) {
            sr[w] = dw;
            amw[w] = aw;
          }
        }
        n_def = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(dcnt)));
        n_amb = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(acnt)));
        __syncwarp();
        if (n_amb > 0) {
          // the ambiguous list, ascending: one word at a time (lane = bit)
          int base = 0;
          for (int w = 0; w < nwords; ++w) {
            const uint32_t bits = amw[w];
            if (bits == 0u) continue;
            const int pos = base + __popc(bits & ((1u << lane) - 1u));
            if (((bits >> lane) & 1u) && pos < kAmbCap) ai[pos] = w * 32 + lane;
            base += __popc(bits);
          }
        }
      } else {
#pragma unroll 4
        for (int j0 = 0; j0 < nb; j0 += 32) {
          const int j = j0 + lane;
          const bool cand = j < nb && is_cand(j);
          const float xv = cand ? ord32_inv(kr[j]) : 0.f;
          const bool def = cand && xv > hi_v;
          const bool amb = cand && !def && xv >= lo_v;
          const unsigned dm = __ballot_sync(0xffffffffu, def);
          const unsigned am = __ballot_sync(0xffffffffu, amb);
          if (lane == 0) sr[j0 / 32] = dm;
          const int pos = n_amb + __popc(am & ((1u << lane) - 1u));
          if (amb && pos < kAmbCap) ai[pos] = j;
          n_def += __popc(dm);
          n_amb += __popc(am);
        }
      }
      __syncwarp();
      const int need = take - n_def;
      if (need < 0 || need > n_amb) {
        report(status, PISA_ERR_DEVICE_CHECK);  // the screening bound did not hold
      } else if (need == n_amb) {
        // every ambiguous candidate is in
        for (int a = lane; a < min(n_amb, kAmbCap); a += 32) atomicOr(&sr[ai[a] / 32], 1u << (ai[a] % 32));
        if (n_amb > kAmbCap)
          for (int j = lane; j < nb; j += 32) {
            const float xv = is_cand(j) ? ord32_inv(kr[j]) : 0.f;
            if (is_cand(j) && xv <= hi_v && xv >= lo_v) atomicOr(&sr[j / 32], 1u << (j % 32));
          }
      } else if (need > 0 && n_amb <= 32) {
        // exact keys (the whole warp on each candidate in turn), lane a keeps
        // candidate a's; rank = keys above + equal keys of lower index
        const bool has = lane < n_amb;
        const int ja = has ? ai[lane] : 0;
        uint64_t ka = 0ull;
        for (int b = 0; b < n_amb; ++b) {
          const int jb = ai[b];
          const uint64_t kb = score_key_warp<D, BIAS>(
              qrow, kh + static_cast<size_t>(jb) * D, scale, mh ? mh[jb] : 0.f, eps, mh != nullptr,
              bon ? bon[static_cast<size_t>(i) * nb + jb] : 0.f, lane);
          if (lane == b) ka = kb;
        }
        int rank = 0;
        for (int b = 0; b < n_amb; ++b) {
          const uint64_t kb = __shfl_sync(0xffffffffu, ka, b);
          const int jb = __shfl_sync(0xffffffffu, ja, b);
          rank += (kb > ka) || (kb == ka && jb < ja);
        }
        if (has && rank < need) atomicOr(&sr[ja / 32], 1u << (ja % 32));
      } else if (need > 0 && n_amb <= kAmbCap) {
        // exact scores of the ambiguous candidates, then their exact top-`need`
        for (int a = lane; a < n_amb; a += 32) ak[a] = exact_key(ai[a]);
        __syncwarp();
        int eq_take;
        const uint64_t kstar = warp_radix_select<64>(
            n_amb, need,
            [&](int a, uint64_t& key) {
              key = ak[a];
              return true;
            },
            hr, lane, &eq_take);
        int eq_seen = 0;
        for (int a0 = 0; a0 < n_amb; a0 += 32) {
          const int a = a0 + lane;
          const uint64_t key = (a < n_amb) ? ak[a] : 0ull;
          const bool gt = a < n_amb && key > kstar;
          const bool eq = a < n_amb && key == kstar;
          const unsigned eqm = __ballot_sync(0xffffffffu, eq);
          const int rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
          if (gt || (eq && rank < eq_take)) atomicOr(&sr[ai[a] / 32], 1u << (ai[a] % 32));
          eq_seen += __popc(eqm);
        }
      } else if (need > 0) {
        // mass near-ties: more ambiguous candidates than the buffer holds; the
        // exact keys are recomputed on every pass of the selection
        auto in_window = [&](int j) {
          if (!is_cand(j)) return false;
          const float xv = ord32_inv(kr[j]);
          return xv <= hi_v && xv >= lo_v;
        };
        int eq_take;
        const uint64_t kstar = warp_radix_select<64>(
            nb, need,
            [&](int j, uint64_t& key) {
              if (!in_window(j)) return false;
              key = exact_key(j);
              return true;
            },
            hr, lane, &eq_take);
        int eq_seen = 0;
        for (int j0 = 0; j0 < nb; j0 += 32) {
          const int j = j0 + lane;
          const bool win = j < nb && in_window(j);
          const uint64_t key = win ? exact_key(j) : 0ull;
          const bool gt = win && key > kstar;
          const bool eq = win && key == kstar;
          const unsigned eqm = __ballot_sync(0xffffffffu, eq);
          const int rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
          if (gt || (eq && rank < eq_take)) atomicOr(&sr[j / 32], 1u << (j % 32));
          eq_seen += __popc(eqm);
        }
      }
    }
    __syncwarp();
    // add the band and the sinks
    for (int j = lo_band + lane; j <= hi_band; j += 32) atomicOr(&sr[j / 32], 1u << (j % 32));
    for (int j = lane; j < n_sink; j += 32) atomicOr(&sr[j / 32], 1u << (j % 32));
    __syncwarp();
    // emit ascending, one bitmask word at a time (lane = bit), pad with -1
    int32_t* out = idx + (static_cast<size_t>(blockIdx.y) * nb + i) * max_sel;
    int written = 0;
#pragma unroll 4
    for (int w = 0; w < nwords; ++w) {
      const uint32_t bits = sr[w];
      if (bits == 0u) continue;
      const int pos = written + __popc(bits & ((1u << lane) - 1u));
      if (((bits >> lane) & 1u) && pos < max_sel) out[pos] = w * 32 + lane;
      written += __popc(bits);
    }
    for (int p = written + lane; p < max_sel; p += 32) out[p] = -1;
    if (lane == 0) cnt[static_cast<size_t>(blockIdx.y) * nb + i] = min(written, max_sel);
    __syncwarp();
  }
}

}  // namespace

int launch_route(const float* qbar, const float* kbar, int heads, int nb, int d, int topk,
                 int band, int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
                 cudaStream_t stream, const float* mnorm, float eps, float scale, int n_sink,
                 const float* bonus) {
  const bool bias = mnorm != nullptr || bonus != nullptr;
  const int nbp = (nb + 3) & ~3;
  // live rows per CTA: as many as kScoreBudget of score rows hold, at most 32;
  // the row layout is the next of 8 / 16 / 32, halved while the grid would
  // not cover the GPU
  int R = static_cast<int>(kScoreBudget / (4 * static_cast<size_t>(nbp)));
  R = max(1, min(32, R));
  int RL = R > 16 ? 32 : (R > 8 ? 16 : 8);
  while (RL > 8 && static_cast<long long>(ceil_div(nb, R)) * heads < 2 * 148) {
    RL /= 2;
    R = min(R, RL);
  }
  const size_t smem = static_cast<size_t>(RL) * d * 4 + static_cast<size_t>(kChunkFloats) * 4 +
                      static_cast<size_t>(R) * nbp * 4 +
                      static_cast<size_t>(kWarps) * ceil_div(nb, 32) * 4 +
                      (bias ? static_cast<size_t>(nb) * 4 : 0);
  dim3 grid(ceil_div(nb, R), heads);
  auto run = [&](auto kern) -> int {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
    kern<<<grid, kThreads, smem, stream>>>(qbar, kbar, nb, R, topk, band, idx, cnt, max_sel,
                                           mnorm, eps, scale, dev_status, min(n_sink, nb), bonus);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  auto pick = [&](auto d_tag, auto b_tag) -> int {
    constexpr int DD = decltype(d_tag)::value;
    constexpr bool BB = decltype(b_tag)::value;
    if (RL == 32) return run(route_kernel<DD, BB, 32>);
    if (RL == 16) return run(route_kernel<DD, BB, 16>);
    return run(route_kernel<DD, BB, 8>);
  };
  using D128 = std::integral_constant<int, 128>;
  using D64 = std::integral_constant<int, 64>;
  if (d == 128) return bias ? pick(D128{}, std::true_type{}) : pick(D128{}, std::false_type{});
  return bias ? pick(D64{}, std::true_type{}) : pick(D64{}, std::false_type{});
}

}  // namespace pisa
