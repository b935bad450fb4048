// Block routing: S_i = band(i) U top-k{ j outside the band } by the pooled
// score s * qbar_i . kbar_j, lower block index first among equal scores.
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Figure 4 "Prepare Phase" and Algorithm 1 step 2; the band as
// in the Piecewise-Taylor-Attention README ("Knobs", band=b).
//
// Since s > 0, the ranking is that of x_ij = qbar_i . kbar_j. Each x_ij is a
// double-float dot product (error-free products and sums, about 2^-44
// relative), mapped to a 64-bit key whose integer order is the value order.
// A CTA owns R query blocks of one head:
//   phase A: every thread walks its key blocks j and accumulates R
//            independent double-float dot products (R-way ILP), storing the
//            keys in shared memory;
//   phase B: warp r selects for row r with an 8-pass radix select (8-bit
//            digits, warp-aggregated shared-memory histograms) that finds the
//            k-th largest key K*; keys above K* are taken, and among keys
//            equal to K* the lowest block indices are taken, which is the
//            lowest-index tie-break. The band is added and the set is emitted
//            in ascending order with ballots.
#include "common.cuh"
#include "kernels.h"

namespace pisa {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = 8;
constexpr size_t kKeyBudget = 131072;  // bytes of shared memory for keys

__device__ __forceinline__ int digit_of(uint64_t key, int shift) {
  return static_cast<int>((key >> shift) & 0xffu);
}

template <int D>
__global__ void __launch_bounds__(kThreads)
route_kernel(const float* __restrict__ qbar, const float* __restrict__ kbar, int nb, int R,
             int topk, int band, int32_t* __restrict__ idx, int32_t* __restrict__ cnt,
             int max_sel) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* qs = reinterpret_cast<float*>(smem_raw);                       // [R][D]
  uint64_t* keys = reinterpret_cast<uint64_t*>(qs + R * D);            // [R][nb]
  uint32_t* hist = reinterpret_cast<uint32_t*>(keys + static_cast<size_t>(R) * nb);  // [R][256]
  uint32_t* selw = hist + R * 256;                                      // [R][nwords]
  const int nwords = ceil_div(nb, 32);

  const int h = blockIdx.y;
  const int i0 = blockIdx.x * R;
  const int rows = min(R, nb - i0);
  const int tid = threadIdx.x;
  const float* qh = qbar + static_cast<size_t>(h) * nb * D;
  const float* kh = kbar + static_cast<size_t>(h) * nb * D;

  for (int e = tid; e < rows * D; e += kThreads) qs[e] = qh[static_cast<size_t>(i0) * D + e];
  __syncthreads();

  // ---- phase A: double-float scores -------------------------------------
  for (int j = tid; j < nb; j += kThreads) {
    DFloat acc[kMaxRows];
    const float4* kr = reinterpret_cast<const float4*>(kh + static_cast<size_t>(j) * D);
#pragma unroll 4
    for (int c4 = 0; c4 < D / 4; ++c4) {
      const float4 kv = __ldg(kr + c4);
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < rows) {
          const float4 qv = *reinterpret_cast<const float4*>(qs + r * D + 4 * c4);
          acc[r].fma_acc(qv.x, kv.x);
          acc[r].fma_acc(qv.y, kv.y);
          acc[r].fma_acc(qv.z, kv.z);
          acc[r].fma_acc(qv.w, kv.w);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
      if (r < rows) keys[static_cast<size_t>(r) * nb + j] = dfloat_key(acc[r].hi, acc[r].lo);
  }
  __syncthreads();

  // ---- phase B: per-row selection (warp r <-> row i0 + r) -----------------
  const int warp = tid / 32, lane = tid % 32;
  for (int r = warp; r < rows; r += kThreads / 32) {
    const int i = i0 + r;
    const uint64_t* kr = keys + static_cast<size_t>(r) * nb;
    uint32_t* hr = hist + r * 256;
    uint32_t* sr = selw + r * nwords;
    const int lo_band = max(0, i - band), hi_band = min(nb - 1, i + band);
    const int n_cand = nb - (hi_band - lo_band + 1);
    const int take = min(topk, n_cand);

    for (int w = lane; w < nwords; w += 32) sr[w] = 0u;
    __syncwarp();

    if (take == n_cand) {
      // every candidate is selected: the whole row
      for (int w = lane; w < nwords; w += 32) {
        const int base = w * 32;
        const int valid = min(32, nb - base);
        sr[w] = (valid == 32) ? 0xffffffffu : ((1u << valid) - 1u);
      }
    } else if (take > 0) {
      uint64_t prefix = 0, pmask = 0;
      int need = take;  // how many still to pick at or below the current prefix
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = lane; b < 256; b += 32) hr[b] = 0u;
        __syncwarp();
        for (int j0 = 0; j0 < nb; j0 += 32) {
          const int j = j0 + lane;
          const bool cand = j < nb && (j < lo_band || j > hi_band);
          const uint64_t key = cand ? kr[j] : 0ull;
          const bool match = cand && ((key & pmask) == prefix);
          const int dg = match ? digit_of(key, shift) : -1;
          const unsigned mm = __ballot_sync(0xffffffffu, match);
          if (mm) {
            const unsigned peers = __match_any_sync(0xffffffffu, dg);
            if (match && (__ffs(peers) - 1) == lane) atomicAdd(&hr[dg], __popc(peers));
          }
        }
        __syncwarp();
        // find the digit holding the need-th largest key: scan bins 255..0
        uint32_t cnt8[8];
        uint32_t mine = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          cnt8[t] = hr[255 - (lane * 8 + t)];
          mine += cnt8[t];
        }
        uint32_t incl = mine;  // inclusive prefix over lanes (descending digits)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - mine;
        int found_digit = -1, above = 0;
        if (excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need)) {
          uint32_t run = excl;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            if (found_digit < 0) {
              if (run + cnt8[t] >= static_cast<uint32_t>(need)) {
                found_digit = 255 - (lane * 8 + t);
                above = static_cast<int>(run);
              } else {
                run += cnt8[t];
              }
            }
          }
        }
        const unsigned who = __ballot_sync(0xffffffffu, found_digit >= 0);
        const int src = __ffs(who) - 1;
        found_digit = __shfl_sync(0xffffffffu, found_digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        prefix |= static_cast<uint64_t>(found_digit) << shift;
        pmask |= 0xffull << shift;
        need -= above;
        __syncwarp();
      }
      // prefix = K*, the take-th largest key; `need` keys equal to K* remain.
      int eq_seen = 0;
      for (int j0 = 0; j0 < nb; j0 += 32) {
        const int j = j0 + lane;
        const bool cand = j < nb && (j < lo_band || j > hi_band);
        const uint64_t key = cand ? kr[j] : 0ull;
        const bool gt = cand && key > prefix;
        const bool eq = cand && key == prefix;
        const unsigned eqm = __ballot_sync(0xffffffffu, eq);
        const int rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
        const bool pick = gt || (eq && rank < need);
        const unsigned pm = __ballot_sync(0xffffffffu, pick);
        if (lane == 0) sr[j0 / 32] = pm;
        eq_seen += __popc(eqm);
      }
    }
    __syncwarp();
    // add the band
    for (int j = lo_band + lane; j <= hi_band; j += 32) atomicOr(&sr[j / 32], 1u << (j % 32));
    __syncwarp();
    // emit ascending, pad with -1
    int32_t* out = idx + (static_cast<size_t>(blockIdx.y) * nb + i) * max_sel;
    int written = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t bits = (w < nwords) ? sr[w] : 0u;
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = written + incl - c;
      uint32_t b = bits;
      while (b) {
        const int t = __ffs(b) - 1;
        b &= b - 1;
        if (pos < max_sel) out[pos] = w * 32 + t;
        ++pos;
      }
      written += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int p = written + lane; p < max_sel; p += 32) out[p] = -1;
    if (lane == 0) cnt[static_cast<size_t>(blockIdx.y) * nb + i] = min(written, max_sel);
    __syncwarp();
  }
}

}  // namespace

int launch_route(const float* qbar, const float* kbar, int heads, int nb, int d, int topk,
                 int band, int32_t* idx, int32_t* cnt, int max_sel, int32_t* dev_status,
                 cudaStream_t stream) {
  (void)dev_status;
  int R = static_cast<int>(kKeyBudget / (8 * static_cast<size_t>(nb)));
  R = max(1, min(kMaxRows, R));
  const int nwords = ceil_div(nb, 32);
  const size_t smem = static_cast<size_t>(R) * nb * 8 + static_cast<size_t>(R) * d * 4 +
                      static_cast<size_t>(R) * 256 * 4 + static_cast<size_t>(R) * nwords * 4;
  dim3 grid(ceil_div(nb, R), heads);
  auto run = [&](auto kern) -> int {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)));
    kern<<<grid, kThreads, smem, stream>>>(qbar, kbar, nb, R, topk, band, idx, cnt, max_sel);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  return d == 128 ? run(route_kernel<128>) : run(route_kernel<64>);
}

}  // namespace pisa
