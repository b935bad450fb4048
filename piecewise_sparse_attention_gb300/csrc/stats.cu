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
//
// Without H (the hot path) `block_means_kernel` issues every 16-byte load of
// the requested tensors before any arithmetic, so a CTA has all of its block
// in flight at once, and merges the partial sums in one pass (shuffles within
// a warp, then one shared-memory step across warps). With H, bf16 inputs with
// d = 128 and kbar requested take the means kernel and then H_j on the tensor
// cores (launch_block_h_tc: the exact three-term split of the centred keys,
// float32 accumulation, centred on the kbar just written); other inputs, and H
// without kbar, take the staged `block_stats_kernel`, which keeps the rows in
// shared memory for the d x d product on the CUDA cores.
#include "common.cuh"
#include "kernels.h"
#include "rowops.cuh"
#include "tc_ptx.cuh"

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

// Means / sums of up to three tensors of one 64-row block (no H).
struct MeansArgs {
  const void* src[3];
  float* dst[3];
  int is_sum[3];  // 1: plain sum (Vhat), 0: mean over the block's rows
};

// Bounded mbarrier waits give up after about a second of SM clock.
constexpr long long kMeansWaitLimit = 2000000000LL;

// Packed TwoSum on float pairs: value = s + c per lane, c collecting the
// exact rounding error of every addition (Knuth's TwoSum, with a - b taken
// as fma(b, -1, a), which rounds exactly like a subtraction).
struct CSum2 {
  uint64_t s = 0, c = 0;
  __device__ __forceinline__ void add(uint64_t x) {
    const uint64_t m1 = f2f(-1.f, -1.f);
    const uint64_t t = add2(s, x);
    const uint64_t bp = fma2(s, m1, t);   // t - s
    const uint64_t ap = fma2(bp, m1, t);  // t - bp
    const uint64_t e = add2(fma2(ap, m1, s), fma2(bp, m1, x));  // (s - ap) + (x - bp)
    s = t;
    c = add2(c, e);
  }
};

// Register caps without spills: five CTAs per SM for one or two tensors
// (48 registers), three for three tensors.
template <typename T, int D, int NT>
__global__ void __launch_bounds__(kThreads, NT < 3 ? 5 : 3)
block_means_kernel(MeansArgs a, int n, int nb, int32_t* status) {
  constexpr int CH = Chunk<T>::kElems;     // channels per 16-byte chunk
  constexpr int NCHUNK = D / CH;           // chunks per row
  constexpr int NG = kThreads / NCHUNK;    // row groups
  constexpr int RPT = kBlock / NG;         // rows per thread
  constexpr int NW = kThreads / 32;
  constexpr int ROWB = D * static_cast<int>(sizeof(T));
  constexpr int TILE = kBlock * ROWB;      // bytes of one tensor's block
  static_assert(RPT * NG == kBlock && 32 % NCHUNK == 0, "layout");
  static_assert(2 * NW * D * 4 <= TILE, "each tensor's partials fit in its tile");
  extern __shared__ __align__(128) uint8_t tiles[];  // [NT][64][D] of T
  __shared__ __align__(8) uint64_t bar;

  const int j = blockIdx.x;
  const int h = blockIdx.y;
  const int row0 = j * kBlock;
  const int nj = min(kBlock, n - row0);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int chunk = tid % NCHUNK;
  const int grp = tid / NCHUNK;

  // one bulk copy per tensor: the block's rows are contiguous in [heads, n, d]
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = static_cast<uint32_t>(nj) * ROWB;
    tc::mbar_arrive_expect_tx(&bar, NT * bytes);
    const size_t off = (static_cast<size_t>(h) * n + row0) * D;
#pragma unroll
    for (int t = 0; t < NT; ++t)
      tc::bulk_load(tiles + t * TILE, static_cast<const T*>(a.src[t]) + off, bytes, &bar);
  }
  int zero = 0;
  const bool got = tc::mbar_wait(&bar, 0, &zero, kMeansWaitLimit);
  if (__syncthreads_or(!got)) {  // CTA-uniform: every thread leaves together
    if (tid == 0) report(status, PISA_ERR_TIMEOUT);
    tc::mbar_wait(&bar, 0, &zero, kMeansWaitLimit);  // the copies may still write
    return;
  }

  uint64_t ps_[NT][CH / 2], pc_[NT][CH / 2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    CSum2 acc[CH / 2];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int row = grp + r * NG;
      if (row < nj) {
        const uint4 u = *reinterpret_cast<const uint4*>(tiles + t * TILE + row * ROWB + chunk * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if constexpr (CH == 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i].add(f2(w[i] << 16, w[i] & 0xffff0000u));
        } else {
#pragma unroll
          for (int i = 0; i < 2; ++i) acc[i].add(f2(w[2 * i], w[2 * i + 1]));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) {
      ps_[t][i] = acc[i].s;
      pc_[t][i] = acc[i].c;
    }
  }
  __syncthreads();  // every tile read: the partials below overwrite the tiles
  float* ps = reinterpret_cast<float*>(tiles);    // [NT][NW][D]
  float* pc = ps + NT * NW * D;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) {
      CSum lo, hi;
      unf2(ps_[t][i], lo.s, hi.s);
      unf2(pc_[t][i], lo.c, hi.c);
      // the row groups of one warp hold the same chunk NCHUNK lanes apart
#pragma unroll
      for (int off = NCHUNK; off < 32; off *= 2) {
        CSum o;
        o.s = __shfl_xor_sync(0xffffffffu, lo.s, off);
        o.c = __shfl_xor_sync(0xffffffffu, lo.c, off);
        lo.merge(o);
        o.s = __shfl_xor_sync(0xffffffffu, hi.s, off);
        o.c = __shfl_xor_sync(0xffffffffu, hi.c, off);
        hi.merge(o);
      }
      if (lane < NCHUNK) {
        const int c = (t * NW + warp) * D + chunk * CH + 2 * i;
        ps[c] = lo.s;
        ps[c + 1] = hi.s;
        pc[c] = lo.c;
        pc[c + 1] = hi.c;
      }
    }
  }
  __syncthreads();
  // one pass over (tensor, channel): the warps' partials merged in warp order
  for (int e = tid; e < NT * D; e += kThreads) {
    const int t = e / D, c = e % D;
    CSum tot;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      CSum part;
      part.s = ps[(t * NW + w) * D + c];
      part.c = pc[(t * NW + w) * D + c];
      tot.merge(part);
    }
    const float sum = tot.value();
    // select instead of indexing the parameter arrays by a run-time t
    float* dst = t == 0 ? a.dst[0] : (t == 1 ? a.dst[1] : a.dst[2]);
    const int is_sum = t == 0 ? a.is_sum[0] : (t == 1 ? a.is_sum[1] : a.is_sum[2]);
    dst[(static_cast<size_t>(h) * nb + j) * D + c] =
        is_sum ? sum : __fdiv_rn(sum, static_cast<float>(nj));
  }
}

template <typename T, int D, int NT>
int launch_means_nt(const MeansArgs& a, int heads, int n, int32_t* status, cudaStream_t stream) {
  constexpr int smem = NT * kBlock * D * static_cast<int>(sizeof(T));
  auto kern = block_means_kernel<T, D, NT>;
  if (smem + 1024 > 48 * 1024) {  // the opt-in covers the static mbarrier too
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  }
  const dim3 grid(ceil_div(n, kBlock), heads);
  kern<<<grid, kThreads, smem, stream>>>(a, n, static_cast<int>(grid.x), status);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

template <typename T, int D>
int launch_means(const void* q, const void* k, const void* v, int heads, int n, float* qbar,
                 float* kbar, float* vsum, int32_t* status, cudaStream_t stream) {
  MeansArgs a{};
  int nt = 0;
  const void* srcs[3] = {q, k, v};
  float* dsts[3] = {qbar, kbar, vsum};
  for (int i = 0; i < 3; ++i) {
    if (dsts[i] == nullptr) continue;
    a.src[nt] = srcs[i];
    a.dst[nt] = dsts[i];
    a.is_sum[nt] = (i == 2);
    ++nt;
  }
  if (nt == 0) return PISA_OK;
  if (nt == 1) return launch_means_nt<T, D, 1>(a, heads, n, status, stream);
  if (nt == 2) return launch_means_nt<T, D, 2>(a, heads, n, status, stream);
  return launch_means_nt<T, D, 3>(a, heads, n, status, stream);
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
                       int h_bf16, int32_t* status, cudaStream_t stream) {
  const bool wh = hmat != nullptr;
  if (wh && in_bf16 && d == 128 && kbar != nullptr) {
    // the means first, then H_j on the tensor cores from the kbar just written
    const int rc = launch_means<__nv_bfloat16, 128>(q, k, v, heads, n, qbar, kbar, vsum, status,
                                                     stream);
    if (rc != PISA_OK) return rc;
    return launch_block_h_tc(k, v, heads, n, kbar, hmat, h_bf16, status, stream);
  }
#define PISA_STATS_CASE(T, D)                                                                  \
  return wh ? launch<T, D, true>(q, k, v, heads, n, qbar, kbar, vsum, hmat, h_bf16, stream)    \
            : launch_means<T, D>(q, k, v, heads, n, qbar, kbar, vsum, status, stream)
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
