// Global first-order statistic of the hybrid approximation:
//   Hbar = (1/n_b) sum_j H_j = (1/n_b) (K^T V - sum_j kbar_j (x) Vhat_j),
// with H_j = sum_n (k_{j,n} - kbar_j)^T v_{j,n} ("PISA: Piecewise Sparse
// Attention Is Wiser for Efficient Diffusion Transformers", Section 3.3 Eq. 10
// and Appendix C "Notation"; the identity is the one the
// Piecewise-Taylor-Attention README uses for its "hc-free" statistics).
//
// The token range of a head is split over `splits` CTAs; each CTA forms its
// part of K^T V and subtracts the kbar_j (x) Vhat_j of the blocks it covers.
// The head's CTAs (at most 8) form one thread-block cluster and sum their
// partials in rank order through distributed shared memory: deterministic,
// no atomics, no zeroing.
//   bf16, d = 128: K^T V on tcgen05 (A = K read MN-major, i.e. transposed,
//                  B = V MN-major, f32 accumulator in TMEM), 64-token tiles
//                  through a 2-stage TMA ring;
//   otherwise:     float32 CUDA-core product.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace pisa {
namespace {

constexpr long long kWait = 2000000000LL;

// thread-block cluster helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_cluster(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             int32_t* status, long long limit) {
  if (tc::mbar_wait(bar, parity, abort, limit)) return true;
  if (!*abort) {
    *abort = 1;
    report(status, PISA_ERR_TIMEOUT);
  }
  return false;
}

// ---------------------------------------------------------------------------
// tcgen05 path (bf16, d = 128)
// ---------------------------------------------------------------------------
constexpr int GD = 128;
constexpr int GT = 64;                  // tokens per tile (one block)
constexpr int G_PANEL = GT * 128;       // [64 tokens][64 channels] bf16 = 8 KB
constexpr int G_TILE = 2 * G_PANEL;     // [64 tokens][128 channels] = 16 KB
constexpr int G_STAGES = 2;
constexpr int G_THREADS = 128;

__global__ void __launch_bounds__(G_THREADS)
global_h_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, int n, int nb, int splits,
                   const float* __restrict__ kbar, const float* __restrict__ vsum,
                   float* __restrict__ hbar, int32_t* status) {
  extern __shared__ unsigned char raw[];
  unsigned char* smem = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
  unsigned char* sK = smem;                                // stages x 16 KB
  unsigned char* sV = smem + G_STAGES * G_TILE;            // stages x 16 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * G_STAGES * G_TILE);
  uint64_t* full = bars;                 // [stage]
  uint64_t* empty = bars + G_STAGES;     // [stage]
  uint64_t* done = bars + 2 * G_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * G_STAGES + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int h = blockIdx.y, sp = blockIdx.x;
  const int t0 = static_cast<int>((static_cast<long long>(nb) * sp) / splits);
  const int t1 = static_cast<int>((static_cast<long long>(nb) * (sp + 1)) / splits);
  const int T = t1 - t0;  // tiles = blocks of this CTA

  if (tid == 0) {
    *abort = 0;
    for (int s = 0; s < G_STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0 && T > 0) {
    // single thread: TMA one tile ahead of the MMAs
    constexpr uint32_t IDESC = tc::idesc_bf16_f32(GD, GD, true) | (1u << 15);  // A, B MN-major
    auto load = [&](int i) {
      const int s = i % G_STAGES;
      tc::mbar_arrive_expect_tx(&full[s], 2 * G_TILE);
      for (int p = 0; p < 2; ++p) {
        tc::tma_load_3d(sK + s * G_TILE + p * G_PANEL, &map_k, 64 * p, (t0 + i) * GT, h, &full[s]);
        tc::tma_load_3d(sV + s * G_TILE + p * G_PANEL, &map_v, 64 * p, (t0 + i) * GT, h, &full[s]);
      }
    };
    bool ok = true;
    load(0);
    for (int i = 0; i < T && ok; ++i) {
      if (i + 1 < T) {
        if (i + 1 >= G_STAGES)
          ok = wait_bounded(&empty[(i + 1) % G_STAGES], ((i + 1) / G_STAGES - 1) & 1, abort,
                            status, kWait);
        if (!ok) break;
        load(i + 1);
      }
      const int s = i % G_STAGES;
      if (!(ok = wait_bounded(&full[s], (i / G_STAGES) & 1, abort, status, kWait))) break;
      tc::tc_fence_after();
      const uint32_t ka = tc::smem_u32(sK + s * G_TILE), va = tc::smem_u32(sV + s * G_TILE);
#pragma unroll
      for (int ks = 0; ks < GT / 16; ++ks)
        tc::mma_ss(tmem, tc::smem_desc_sw128(ka + ks * 2048, G_PANEL, 1024),
                   tc::smem_desc_sw128(va + ks * 2048, G_PANEL, 1024), IDESC,
                   (i > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(done);
    if (!ok) {
      // drain the copies this thread started
      int zero = 0;
      for (int s = 0; s < G_STAGES; ++s) tc::mbar_wait(&full[s], 0, &zero, kWait);
    }
  }
  bool ok = T > 0;
  if (ok) ok = wait_bounded(done, 0, abort, status, kWait);
  // one decision for the whole CTA: the epilogue below has block barriers
  ok = __syncthreads_and(ok && !*abort) != 0;
  tc::tc_fence_after();
  // thread <-> key channel c (TMEM lane): its row of K^T V from TMEM, minus
  // sum_j kbar_j[c] Vhat_j over this CTA's blocks. kbar and Vhat of up to
  // kChunk blocks at a time are staged in the (now idle) stage buffers with
  // coalesced loads, so the row update reads shared memory.
  constexpr int kChunk = 32;
  float* s_kb = reinterpret_cast<float*>(smem);  // [kChunk][GD]
  float* s_vs = s_kb + kChunk * GD;               // [kChunk][GD]
  const int c = warp * 32 + lane;
  const float inv_nb = 1.f / static_cast<float>(nb);
  const float* kb = kbar + (static_cast<size_t>(h) * nb) * GD;
  const float* vs = vsum + (static_cast<size_t>(h) * nb) * GD;
  float g[GD];
  if (ok) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * q4, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) g[32 * q4 + e] = __uint_as_float(r[e]);
    }
  }
  for (int j0 = t0; j0 < t1 && ok; j0 += kChunk) {
    const int m = min(kChunk, t1 - j0);
    __syncthreads();  // the stage buffers (and the previous chunk) are free
    for (int e = tid; e < m * (GD / 4); e += G_THREADS) {
      const int jj = e / (GD / 4), c4 = e % (GD / 4);
      reinterpret_cast<float4*>(s_kb)[jj * (GD / 4) + c4] =
          __ldg(reinterpret_cast<const float4*>(kb + static_cast<size_t>(j0 + jj) * GD) + c4);
      reinterpret_cast<float4*>(s_vs)[jj * (GD / 4) + c4] =
          __ldg(reinterpret_cast<const float4*>(vs + static_cast<size_t>(j0 + jj) * GD) + c4);
    }
    __syncthreads();
    for (int jj = 0; jj < m; ++jj) {
      const float kc = s_kb[jj * GD + c];
      const float4* vr = reinterpret_cast<const float4*>(s_vs + jj * GD);
#pragma unroll
      for (int e4 = 0; e4 < GD / 4; ++e4) {
        const float4 vv = vr[e4];
        g[4 * e4 + 0] = fmaf(-kc, vv.x, g[4 * e4 + 0]);
        g[4 * e4 + 1] = fmaf(-kc, vv.y, g[4 * e4 + 1]);
        g[4 * e4 + 2] = fmaf(-kc, vv.z, g[4 * e4 + 2]);
        g[4 * e4 + 3] = fmaf(-kc, vv.w, g[4 * e4 + 3]);
      }
    }
  }
  // Deterministic sum over the head's CTAs (one thread-block cluster): each
  // CTA leaves its partial in its own stage buffers (row c, float4 chunk k at
  // position k ^ (c & 7), so both the row-wise stores and the reads below are
  // free of bank conflicts); after a cluster barrier CTA r sums rows
  // [128 r / splits, 128 (r + 1) / splits) over the cluster's partials in
  // rank order through distributed shared memory. No atomics, no zeroing.
  __syncthreads();  // every read of the staged kbar / Vhat is done
  float4* part = reinterpret_cast<float4*>(smem);  // [GD][GD / 4]
#pragma unroll
  for (int k4 = 0; k4 < GD / 4; ++k4)
    part[c * (GD / 4) + (k4 ^ (c & 7))] =
        ok ? make_float4(g[4 * k4], g[4 * k4 + 1], g[4 * k4 + 2], g[4 * k4 + 3])
           : make_float4(0.f, 0.f, 0.f, 0.f);
  cluster_sync();
  {
    const int rank = static_cast<int>(cluster_ctarank());
    const int rb = GD * rank / splits, re = GD * (rank + 1) / splits;
    const uint32_t local = tc::smem_u32(part);
    for (int it = tid; it < (re - rb) * (GD / 4); it += G_THREADS) {
      const int row = rb + it / (GD / 4), k4 = it % (GD / 4);
      const uint32_t off = static_cast<uint32_t>(row * (GD / 4) + (k4 ^ (row & 7))) * 16u;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < splits; ++r) {
        const float4 x = ld_cluster_f4(map_cluster(local + off, static_cast<uint32_t>(r)));
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      *reinterpret_cast<float4*>(hbar + (static_cast<size_t>(h) * GD + row) * GD + 4 * k4) =
          make_float4(acc.x * inv_nb, acc.y * inv_nb, acc.z * inv_nb, acc.w * inv_nb);
    }
  }
  cluster_sync();  // the partials stay until every CTA of the cluster has read them
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------------------
// CUDA-core path (float32 inputs, or d = 64)
// ---------------------------------------------------------------------------
constexpr int S_THREADS = 256;
constexpr int S_ROWS = 16;  // tokens staged per step

template <typename T, int D>
__global__ void __launch_bounds__(S_THREADS)
global_h_simt_kernel(const T* __restrict__ k, const T* __restrict__ v, int n, int nb, int splits,
                     const float* __restrict__ kbar, const float* __restrict__ vsum,
                     float* __restrict__ hbar) {
  constexpr int TILE = (D == 128) ? 8 : 4;  // TILE x TILE outputs per thread
  constexpr int PER_ROW = D / TILE;         // PER_ROW^2 = S_THREADS
  static_assert(PER_ROW * PER_ROW == S_THREADS, "one output tile per thread");
  extern __shared__ __align__(16) float sh[];
  float* ks = sh;                 // [S_ROWS][D] staged keys
  float* vs = sh + S_ROWS * D;    // [S_ROWS][D] staged values
  const int tid = threadIdx.x;
  const int h = blockIdx.y, sp = blockIdx.x;
  const int j0 = static_cast<int>((static_cast<long long>(nb) * sp) / splits);
  const int j1 = static_cast<int>((static_cast<long long>(nb) * (sp + 1)) / splits);
  const int r0 = j0 * kBlock, r1 = min(n, j1 * kBlock);
  const int c0 = (tid / PER_ROW) * TILE, e0 = (tid % PER_ROW) * TILE;
  const size_t hoff = static_cast<size_t>(h) * n * D;
  float acc[TILE][TILE];
#pragma unroll
  for (int a = 0; a < TILE; ++a)
#pragma unroll
    for (int b = 0; b < TILE; ++b) acc[a][b] = 0.f;
  for (int rb = r0; rb < r1; rb += S_ROWS) {
    __syncthreads();
    for (int e = tid; e < S_ROWS * D; e += S_THREADS) {
      const int rr = e / D, cc = e % D;
      const int row = rb + rr;
      const bool okr = row < r1;
      ks[rr * D + cc] = okr ? static_cast<float>(k[hoff + static_cast<size_t>(row) * D + cc]) : 0.f;
      vs[rr * D + cc] = okr ? static_cast<float>(v[hoff + static_cast<size_t>(row) * D + cc]) : 0.f;
    }
    __syncthreads();
    for (int rr = 0; rr < S_ROWS; ++rr) {
      float kc[TILE], vv[TILE];
#pragma unroll
      for (int a = 0; a < TILE; ++a) kc[a] = ks[rr * D + c0 + a];
#pragma unroll
      for (int b = 0; b < TILE; ++b) vv[b] = vs[rr * D + e0 + b];
#pragma unroll
      for (int a = 0; a < TILE; ++a)
#pragma unroll
        for (int b = 0; b < TILE; ++b) acc[a][b] = fmaf(kc[a], vv[b], acc[a][b]);
    }
  }
  const float inv_nb = 1.f / static_cast<float>(nb);
  for (int j = j0; j < j1; ++j) {
    const float* kb = kbar + (static_cast<size_t>(h) * nb + j) * D;
    const float* vb = vsum + (static_cast<size_t>(h) * nb + j) * D;
#pragma unroll
    for (int a = 0; a < TILE; ++a)
#pragma unroll
      for (int b = 0; b < TILE; ++b) acc[a][b] = fmaf(-kb[c0 + a], vb[e0 + b], acc[a][b]);
  }
  // the head's CTAs (one cluster) sum their partials in rank order, as in the
  // tensor-core kernel: partial row c, float4 chunk q at position q ^ (c & 7)
  __syncthreads();  // every read of the staged tokens is done
  float4* part = reinterpret_cast<float4*>(sh);  // [D][D / 4]
#pragma unroll
  for (int a = 0; a < TILE; ++a)
#pragma unroll
    for (int b = 0; b < TILE; b += 4) {
      const int c = c0 + a, q4 = (e0 + b) / 4;
      part[c * (D / 4) + (q4 ^ (c & 7))] =
          make_float4(acc[a][b], acc[a][b + 1], acc[a][b + 2], acc[a][b + 3]);
    }
  cluster_sync();
  {
    const int rank = static_cast<int>(cluster_ctarank());
    const int rb = D * rank / splits, re = D * (rank + 1) / splits;
    const uint32_t local = tc::smem_u32(part);
    for (int it = tid; it < (re - rb) * (D / 4); it += S_THREADS) {
      const int row = rb + it / (D / 4), q4 = it % (D / 4);
      const uint32_t off = static_cast<uint32_t>(row * (D / 4) + (q4 ^ (row & 7))) * 16u;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < splits; ++r) {
        const float4 x = ld_cluster_f4(map_cluster(local + off, static_cast<uint32_t>(r)));
        sum.x += x.x;
        sum.y += x.y;
        sum.z += x.z;
        sum.w += x.w;
      }
      *reinterpret_cast<float4*>(hbar + (static_cast<size_t>(h) * D + row) * D + 4 * q4) =
          make_float4(sum.x * inv_nb, sum.y * inv_nb, sum.z * inv_nb, sum.w * inv_nb);
    }
  }
  cluster_sync();  // the partials stay until every CTA of the cluster has read them
}

}  // namespace

int launch_global_h(const void* k, const void* v, int in_bf16, int heads, int n, int d,
                    const float* kbar, const float* vsum, float* hbar, int32_t* dev_status,
                    cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  if (in_bf16 && d == GD) {
    // one cluster of `splits` CTAs per head (at most 8, the portable cluster
    // size); the cluster sums its partials itself, so hbar needs no zeroing
    const int splits = max(1, min(min(nb, 8), (3 * 152) / max(1, heads)));
    CUtensorMap mk, mv;
    const uint64_t dims[3] = {static_cast<uint64_t>(GD), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(heads)};
    const uint64_t strides[2] = {static_cast<uint64_t>(GD) * 2, static_cast<uint64_t>(n) * GD * 2};
    const uint32_t box[3] = {64, GT, 1};
    if (!make_tmap_bf16(&mk, k, 3, dims, strides, box) || !make_tmap_bf16(&mv, v, 3, dims, strides, box))
      return PISA_ERR_CUDA;
    const int smem = 2 * G_STAGES * G_TILE + 256 + 1024;
    PISA_CUDA_TRY(cudaFuncSetAttribute(global_h_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, heads);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PISA_CUDA_TRY(cudaLaunchKernelEx(&cfg, global_h_tc_kernel, mk, mv, n, nb, splits, kbar, vsum,
                                     hbar, dev_status));
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  }
  // one cluster of at most 8 CTAs per head, as above
  const int splits = max(1, min(min(nb, 8), (4 * 152) / max(1, heads)));
  auto launch = [&](auto kern, const auto* kk, const auto* vv, int dd) -> int {
    const size_t smem = static_cast<size_t>(dd) * dd * sizeof(float);  // >= the token staging
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, heads);
    cfg.blockDim = dim3(S_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PISA_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, kk, vv, n, nb, splits, kbar, vsum, hbar));
    return PISA_OK;
  };
  using BF = __nv_bfloat16;
  int rc;
  if (in_bf16)
    rc = d == 128 ? launch(global_h_simt_kernel<BF, 128>, static_cast<const BF*>(k),
                           static_cast<const BF*>(v), 128)
                  : launch(global_h_simt_kernel<BF, 64>, static_cast<const BF*>(k),
                           static_cast<const BF*>(v), 64);
  else
    rc = d == 128 ? launch(global_h_simt_kernel<float, 128>, static_cast<const float*>(k),
                           static_cast<const float*>(v), 128)
                  : launch(global_h_simt_kernel<float, 64>, static_cast<const float*>(k),
                           static_cast<const float*>(v), 64);
  if (rc != PISA_OK) return rc;
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace pisa
