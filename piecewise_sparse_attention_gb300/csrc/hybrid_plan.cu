// The plan of the hybrid tensor-core forward (forward_hybrid_tc.cu): which
// two query blocks share a 128-row query tile, and which two tiles share a
// CTA, written as plan[h][c][x] = query block x (0..3) of CTA c of head h.
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Section 3.3 and Algorithm 1 (Phase 3) define what the hybrid
// forward computes for each query block; how the blocks are grouped into
// tiles and CTAs is this implementation's choice and changes no sum.
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace pisa {
namespace {

// Which query blocks share a 128-row query tile, and which two tiles share a
// CTA. The plan decides how much work the kernel does and how evenly it is
// spread; every plan computes the same sums. A row's exact blocks are the
// same for any plan, but which of them share a 128-key tile depends on the
// union they belong to, so two plans can round differently (the online
// softmax takes its maxima and rounds P per tile); the CTA pairing alone
// changes nothing.
//
// Tiles. A tile runs one exact step per two blocks of the union of its two
// query blocks' critical sets, and a block that is critical for only one of
// them still costs both their rows the products. Two query blocks whose
// critical sets overlap most make the smallest union, so the blocks of a head
// are matched greedily by overlap: the pair with the largest overlap first
// (ties: lower block indices first), then the largest among the rest, and so
// on, over the pairs whose indices differ by at most W. The greedy matching is
// computed in rounds of mutual choices: every unmatched block picks its best
// unmatched partner in the window by that same order, and pairs that picked
// each other are matched (the best remaining pair always does, so every round
// that can make progress does; the result is the greedy matching). Blocks
// left over (no unmatched partner within W, or after the last round) pair in
// index order; an odd one out gets a tile of its own. A head whose bitmasks
// and overlaps do not fit in shared memory (W = 0) keeps neighbouring blocks
// 2t and 2t + 1 together.
//
// CTAs. A CTA streams the exact tiles of its two query tiles side by side,
// so its exact phase lasts as long as the longer list, and while one tile has
// work left alone nothing overlaps its softmax with the other tile's
// products. The tiles of each head are sorted by their number of exact tiles
// (largest first, lower tile number first among equal ones) and consecutive
// tiles share a CTA: the two lists of a CTA are then about equally long and
// the longest CTAs start first.
//
// One CTA per head. plan[h][c][x] = query block x (0..3) of CTA c: tile w
// holds blocks x = 2w (rows 0-63 of the tile) and 2w + 1 (rows 64-127); nb
// stands for no block.
constexpr int PAIR_THREADS = 1024;
constexpr int PAIR_TILE_BITS = 13;  // up to 8192 query tiles (n <= 2^20)
constexpr int PAIR_MAX_TILES = 1 << PAIR_TILE_BITS;
static_assert(PAIR_MAX_TILES == kHybridPlanMaxTiles, "tile index field of the sort keys");
constexpr int PAIR_MAX_ROUNDS = 64;
constexpr size_t PAIR_SMEM_LIMIT = 220 * 1024;

__host__ __device__ inline int pair_pow2(int n_tiles) {
  int p = 1;
  while (p < n_tiles) p <<= 1;
  return p;
}

// words of a bitmask row in the matching mode (a power of two covering nb
// bits), 0 where nb is too large to match
int pair_words(int nb) { return nb <= 256 ? 8 : nb <= 512 ? 16 : nb <= 1024 ? 32 : 0; }

// shared memory of the pairing kernel: keys and tile lists, then either the
// matching state (mate, choice, the counts, every bitmask with a row stride
// of NW + 4 words, the overlaps [W][nb]) or, with NW = 0, one bitmask per
// warp
size_t pair_smem_bytes(int nb, int NW, int W) {
  const size_t n_tiles = (nb + 1) / 2, nwords = (nb + 31) / 32;
  const size_t base = (pair_pow2(static_cast<int>(n_tiles)) + 2 * n_tiles) * 4;
  if (NW == 0) return base + static_cast<size_t>(PAIR_THREADS / 32) * nwords * 4;
  return base + 3 * static_cast<size_t>(nb) * 4 + static_cast<size_t>(nb) * (NW + 4) * 4 +
         static_cast<size_t>(nb) * W;
}

// the largest window in {128, 64, 32, 16} whose matching state fits, else 0
int pair_window(int nb, int NW) {
  if (NW == 0) return 0;
  for (int W = 128; W >= 16; W >>= 1)
    if (pair_smem_bytes(nb, NW, W) <= PAIR_SMEM_LIMIT) return W;
  return 0;
}

// The greedy order of pair (a, b), a < b, with overlap v as one integer: a
// larger key comes first (larger overlap, then lower a, then lower b).
__device__ __forceinline__ uint64_t pair_key(int v, int a, int b) {
  return (static_cast<uint64_t>(v) << 32) | (static_cast<uint32_t>(16383 - a) << 14) |
         static_cast<uint32_t>(16383 - b);
}

// OR critical sets qa and qb (qb = nb: none) of head h into bitmask row
// `row` (one warp); every load of a batch is issued before its atomics
__device__ __forceinline__ void pair_add_sets(uint32_t* row, const int32_t* __restrict__ idx,
                                              const int32_t* __restrict__ cnt, int h, int nb,
                                              int max_sel, int qa, int qb, int lane) {
  const size_t ra = static_cast<size_t>(h) * nb + qa, rb = static_cast<size_t>(h) * nb + qb;
  const int ca = min(cnt[ra], max_sel), cb = qb < nb ? min(cnt[rb], max_sel) : 0;
  for (int e0 = 0; e0 < ca || e0 < cb; e0 += 64) {
    int j[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + lane + 32 * (u & 1);
      const bool in = (u < 2) ? e < ca : e < cb;
      j[u] = in ? idx[((u < 2) ? ra : rb) * max_sel + e] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j[u] >= 0 && j[u] < nb) atomicOr(&row[j[u] >> 5], 1u << (j[u] & 31));
  }
}

__device__ __forceinline__ int pair_warp_sum(int u) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
  return u;
}

// sort key of tile t whose union has u blocks
__device__ __forceinline__ uint32_t pair_tile_key(int t, int u) {
  return (1u << 31) | (static_cast<uint32_t>((u + 1) / 2) << PAIR_TILE_BITS) |
         static_cast<uint32_t>(PAIR_MAX_TILES - 1 - t);
}

template <int NW>  // words of a bitmask row; 0: neighbouring blocks, no matching
__global__ void __launch_bounds__(PAIR_THREADS, 1)
pair_tiles_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int nb,
                  int max_sel, int W, int32_t* __restrict__ plan) {
  extern __shared__ __align__(16) uint32_t pair_smem[];  // 16-byte rows for vector loads
  __shared__ int s_count, s_changed;
  const int n_tiles = ceil_div(nb, 2);
  const int n_ctas = ceil_div(n_tiles, 2);
  const int np2 = pair_pow2(n_tiles);
  const int nwords = ceil_div(nb, 32);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int h = blockIdx.x;
  // matching mode: bitmasks [nb][NW + 4] first (16-byte rows), overlaps
  // [W][nb] bytes, then the keys, tile lists and matching state
  constexpr int BS = NW + 4;
  const size_t head = NW > 0 ? static_cast<size_t>(nb) * BS * 4 + static_cast<size_t>(W) * nb : 0;
  uint32_t* key = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(pair_smem) + head);
  int* ta = reinterpret_cast<int*>(key + np2);  // tile t = blocks ta[t] < tb[t] (tb = nb: none)
  int* tb = ta + n_tiles;
  for (int e = tid; e < np2; e += PAIR_THREADS) key[e] = 0u;

  if constexpr (NW > 0) {
    // row stride of NW + 4 words: 16-byte rows for vector loads, and eight
    // consecutive rows (one phase of a 128-bit load) on distinct banks
    uint32_t* bits = pair_smem;                                                        // [nb][BS]
    uint8_t* ovt = reinterpret_cast<uint8_t*>(bits + static_cast<size_t>(nb) * BS);  // [W][nb]
    int* mate = tb + n_tiles;
    int* choice = mate + nb;
    int* counts = choice + nb;
    // ---- bitmasks of every critical set, overlaps within the window ----------
    // The head's lists are one contiguous [nb][max_sel] array: every thread
    // streams through it with 16 loads in flight (the counts are staged first).
    for (int e = tid; e < nb * BS; e += PAIR_THREADS) bits[e] = 0u;
    for (int e = tid; e < nb; e += PAIR_THREADS) {
      mate[e] = -1;
      choice[e] = -1;
      counts[e] = min(cnt[static_cast<size_t>(h) * nb + e], max_sel);
    }
    __syncthreads();
    {
      const int32_t* lst = idx + static_cast<size_t>(h) * nb * max_sel;
      const int total = nb * max_sel;
      for (int e0 = tid; e0 < total; e0 += 16 * PAIR_THREADS) {
        int j[16], b[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int e = e0 + u * PAIR_THREADS;
          b[u] = e < total ? e / max_sel : 0;
          j[u] = (e < total && e - b[u] * max_sel < counts[b[u]]) ? lst[e] : -1;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (j[u] >= 0 && j[u] < nb) atomicOr(&bits[b[u] * BS + (j[u] >> 5)], 1u << (j[u] & 31));
      }
    }
    __syncthreads();
    // thread e takes block e % nb and part e / nb of its window (the window
    // is split so that every thread has work when nb < PAIR_THREADS)
    const int parts = max(1, min(W, PAIR_THREADS / nb));
    for (int e = tid; e < nb * parts; e += PAIR_THREADS) {
      const int i = e % nb, part = e / nb;
      uint4 bi[NW / 4];
#pragma unroll
      for (int w = 0; w < NW / 4; ++w) bi[w] = reinterpret_cast<const uint4*>(bits + i * BS)[w];
      for (int dd = 1 + part * W / parts; dd <= (part + 1) * W / parts; ++dd) {
        const int j = i + dd;
        int v = 0;
        if (j < nb) {
          const uint4* bj = reinterpret_cast<const uint4*>(bits + j * BS);
#pragma unroll
          for (int w = 0; w < NW / 4; ++w) {
            const uint4 y = bj[w];
            v += __popc(bi[w].x & y.x) + __popc(bi[w].y & y.y) + __popc(bi[w].z & y.z) +
                 __popc(bi[w].w & y.w);
          }
        }
        ovt[(dd - 1) * nb + i] = static_cast<uint8_t>(min(v, 255));
      }
    }
    __syncthreads();
    // ---- greedy matching by rounds of mutual choices --------------------------
    // choice[i]: block i's best unmatched partner (-1: to be found, -2: none
    // left). Partners only ever drop out, so a choice stays the best until
    // that partner is matched; only then is it searched again, by a whole
    // warp. The counts are no longer needed: `counts` lists the searches.
    int* todo = counts;
    auto search = [&](int i) {
      uint64_t best = 0;
      int bj = -1;
#pragma unroll 4
      for (int c = lane; c < 2 * W; c += 32) {
        const int dd = (c >> 1) + 1;
        const int j = (c & 1) ? i - dd : i + dd;
        if (j >= 0 && j < nb && mate[j] < 0) {
          const int lo = min(i, j), hi = max(i, j);
          const uint64_t kk = pair_key(ovt[(dd - 1) * nb + lo], lo, hi);
          if (kk > best) {
            best = kk;
            bj = j;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
        if (ob > best) {
          best = ob;
          bj = oj;
        }
      }
      return bj;
    };
    for (int round = 0; round < PAIR_MAX_ROUNDS; ++round) {
      if (tid == 0) {
        s_count = 0;
        s_changed = 0;
      }
      __syncthreads();
      // list the unmatched blocks whose choice is missing or taken
      for (int b0 = warp * 32; b0 < nb; b0 += PAIR_THREADS) {
        const int i = b0 + lane;
        bool need = false;
        if (i < nb && mate[i] < 0) {
          const int c = choice[i];
          need = c == -1 || (c >= 0 && mate[c] >= 0);
        }
        const unsigned m = __ballot_sync(0xffffffffu, need);
        int pos = 0;
        if (lane == 0 && m) pos = atomicAdd(&s_count, __popc(m));
        pos = __shfl_sync(0xffffffffu, pos, 0);
        if (need) todo[pos + __popc(m & ((1u << lane) - 1u))] = i;
      }
      __syncthreads();
      const int nsearch = s_count;
      for (int e = warp; e < nsearch; e += PAIR_THREADS / 32) {
        const int i = todo[e];
        const int j = search(i);
        if (lane == 0) choice[i] = j >= 0 ? j : -2;
      }
      __syncthreads();
      for (int i = tid; i < nb; i += PAIR_THREADS) {
        const int j = choice[i];
        if (mate[i] < 0 && j >= 0 && choice[j] == i) {
          mate[i] = j;
          s_changed = 1;
        }
      }
      __syncthreads();
      const int changed = s_changed;
      __syncthreads();
      if (!changed) break;
    }
    // ---- leftovers in index order, then the tile list (by lower block) -------
    if (warp == 0) {
      int pending = -1;
      for (int b0 = 0; b0 < nb; b0 += 32) {
        const int i = b0 + lane;
        unsigned m = __ballot_sync(0xffffffffu, i < nb && mate[i] < 0);
        while (m) {
          const int v = b0 + __ffs(m) - 1;
          m &= m - 1;
          if (pending < 0) {
            pending = v;
          } else {
            if (lane == 0) {
              mate[pending] = v;
              mate[v] = pending;
            }
            pending = -1;
          }
        }
        __syncwarp();
      }
      if (pending >= 0 && lane == 0) mate[pending] = nb;
      __syncwarp();
      int t0 = 0;
      for (int b0 = 0; b0 < nb; b0 += 32) {
        const int i = b0 + lane;
        const bool lead = i < nb && mate[i] > i;
        const unsigned m = __ballot_sync(0xffffffffu, lead);
        if (lead) {
          const int t = t0 + __popc(m & ((1u << lane) - 1u));
          ta[t] = i;
          tb[t] = mate[i];
        }
        t0 += __popc(m);
      }
    }
    __syncthreads();
    // ---- exact tiles of every tile ----------------------------------------
    for (int t = warp; t < n_tiles; t += PAIR_THREADS / 32) {
      const uint32_t* ba = bits + ta[t] * BS;
      const uint32_t* bb = tb[t] < nb ? bits + tb[t] * BS : ba;
      int u = 0;
      for (int e = lane; e < nwords; e += 32) u += __popc(ba[e] | bb[e]);
      u = pair_warp_sum(u);
      if (lane == 0) key[t] = pair_tile_key(t, u);
    }
  } else {
    // ---- neighbouring blocks; each warp counts a tile's union in its bitmask -
    uint32_t* wb = reinterpret_cast<uint32_t*>(tb + n_tiles) + warp * nwords;
    __syncthreads();
    for (int t = warp; t < n_tiles; t += PAIR_THREADS / 32) {
      for (int e = lane; e < nwords; e += 32) wb[e] = 0u;
      __syncwarp();
      pair_add_sets(wb, idx, cnt, h, nb, max_sel, 2 * t, 2 * t + 1 < nb ? 2 * t + 1 : nb, lane);
      __syncwarp();
      int u = 0;
      for (int e = lane; e < nwords; e += 32) u += __popc(wb[e]);
      u = pair_warp_sum(u);
      if (lane == 0) {
        ta[t] = 2 * t;
        tb[t] = 2 * t + 1 < nb ? 2 * t + 1 : nb;
        key[t] = pair_tile_key(t, u);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // ---- tiles by decreasing exact tiles: bitonic sort of key[0, np2) ----------
  for (int k = 2; k <= np2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < np2; i += PAIR_THREADS) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t a = key[i], b = key[l];
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            key[i] = b;
            key[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int e = tid; e < 4 * n_ctas; e += PAIR_THREADS) {
    const int slot = e >> 1;  // sorted position of the tile
    const uint32_t kk = slot < np2 ? key[slot] : 0u;
    int qb = nb;
    if (kk >> 31) {
      const int t = PAIR_MAX_TILES - 1 - static_cast<int>(kk & (PAIR_MAX_TILES - 1));
      qb = (e & 1) ? tb[t] : ta[t];
    }
    plan[static_cast<size_t>(h) * 4 * n_ctas + e] = qb;
  }
}

template <int NW>
int launch_pair(const int32_t* idx, const int32_t* cnt, int heads, int nb, int max_sel, int W,
                int32_t* plan, cudaStream_t stream) {
  const size_t bytes = pair_smem_bytes(nb, NW, W);
  if (bytes > 48 * 1024)
    PISA_CUDA_TRY(cudaFuncSetAttribute(pair_tiles_kernel<NW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes)));
  pair_tiles_kernel<NW><<<heads, PAIR_THREADS, bytes, stream>>>(idx, cnt, nb, max_sel, W, plan);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace

int launch_hybrid_plan(const int32_t* idx, const int32_t* cnt, int heads, int nb, int max_sel,
                       int32_t* plan, cudaStream_t stream) {
  // the matching mode indexes the head's [nb][max_sel] lists with 32-bit
  // integers
  int NW = static_cast<long long>(nb) * max_sel <= INT32_MAX ? pair_words(nb) : 0;
  const int W = pair_window(nb, NW);
  if (W == 0) NW = 0;
  switch (NW) {
    case 8: return launch_pair<8>(idx, cnt, heads, nb, max_sel, W, plan, stream);
    case 16: return launch_pair<16>(idx, cnt, heads, nb, max_sel, W, plan, stream);
    case 32: return launch_pair<32>(idx, cnt, heads, nb, max_sel, W, plan, stream);
    default: return launch_pair<0>(idx, cnt, heads, nb, max_sel, 0, plan, stream);
  }
}

}  // namespace pisa
