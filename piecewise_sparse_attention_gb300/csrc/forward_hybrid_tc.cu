// Hybrid-order forward on the tensor cores (tcgen05 + TMEM + TMA), bf16
// inputs, head dim 64 or 128 (template parameter D; a [128][D] tile is D / 64
// swizzled panels).
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Section 3.3 Eq. 9-10 and Algorithm 1 (Phases 1-3): for query
// t of query block i, alpha_tj = e^{q'.kbar_j},
//   D_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} + sum_{j not in S_i} n_j alpha_tj
//   N_t = sum_{j in S_i} sum_n e^{q'.k_{j,n}} v_{j,n} + sum_{j not in S_i} alpha_tj Vhat_j
//         + (sum_{j not in S_i} alpha_tj) q' Hbar.
//
// CTA = two 128-row query tiles of one head, each made of two query blocks
// that need not be neighbours (rows 0-63 and 64-127 of the tile), with the
// same warp roles, TMEM map and MMA issue order as the block-wise kernel
// (forward_tc.cu), over a sequence of "tiles":
//   exact tiles  - per 128-row query tile, the union of its two query
//                  blocks' critical sets, taken two 64-key blocks at a time;
//                  TMA gathers each block into one half of a 128-key K/V tile.
//                  A block that is critical for only one of the two query
//                  blocks gets P = 0 in the other (which sees it through its
//                  centroid below). The two query tiles stream their own
//                  tiles, interleaved on the K and V rings; a tile whose list
//                  is shorter simply idles for the remaining exact steps;
//   centroid tiles - 128 key centroids at a time: S = Q (Kbar_hi + Kbar_lo)^T,
//                  P = alpha masked on the critical blocks, O += P (Vhat_hi +
//                  Vhat_lo); kbar and Vhat are split into bf16 hi + lo parts
//                  (about 16 significant bits), so centroid logits keep
//                  ~2^-17 relative accuracy;
//   first order  - Q (Hbar_hi + Hbar_lo) into the free S columns; the epilogue
//                  forms o = (O + s * tail * Q Hbar) / l, tail = sum of alpha.
// The bf16 hi/lo operands are written into the caller's workspace by a small
// conversion kernel launched first on the same stream, and a pairing kernel
// decides which query blocks share a tile and which tiles share a CTA
// (hybrid_plan.cu).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "rowops.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace pisa {
namespace {

constexpr int TILE_M = 128;
constexpr int TILES = 2;
constexpr int CTA_ROWS = TILE_M * TILES;
constexpr int STAGES = 2;
constexpr int PANEL = 128 * 128;          // [128 rows][64 bf16]
constexpr int HALF_PANEL = 64 * 128;      // [64 rows][64 bf16]
constexpr int NUM_THREADS = 320;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr long long WAIT_LIMIT = 2000000000LL;
constexpr float LAZY = 20.0f;

// a [128 rows][D] tile is D / 64 swizzled panels
template <int D>
struct Smem {
  static constexpr int TILE_BYTES = D / 64 * PANEL;
  static constexpr int Q = 0;
  static constexpr int K = Q + TILES * TILE_BYTES;
  static constexpr int V = K + STAGES * TILE_BYTES;
  static constexpr int BAR = V + STAGES * TILE_BYTES;
  static constexpr int NBAR = 20;
  static constexpr int MISC = BAR + NBAR * 8;   // tmem slot, abort flag, union size
  static constexpr int MASK = MISC + 64;        // route bitmasks [4], unions [2], union lists
};

enum {
  B_Q = 0,
  B_KFULL = 1,
  B_KEMPTY = 3,
  B_VFULL = 5,
  B_VEMPTY = 7,
  B_SFULL = 9,
  B_PFULL = 11,  // +2*tile+half
  B_OFULL = 15,
  B_DRAIN = 17
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int32_t* status) {
  if (tc::mbar_wait(bar, parity, abort, WAIT_LIMIT)) return true;
  if (!*abort) {
    *abort = 1;
    report(status, PISA_ERR_TIMEOUT);
  }
  return false;
}

// Centroid columns that count for a query block: column i <-> block jw + i,
// counted when the block exists and is not in the block's critical set.
__device__ __forceinline__ uint32_t centroid_cols(const uint32_t* mask, int jw, int nb) {
  if (jw >= nb) return 0u;
  const uint32_t valid = (nb - jw >= 32) ? 0xffffffffu : ((1u << (nb - jw)) - 1u);
  return valid & ~mask[jw >> 5];
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
forward_hybrid_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_kb,
                         const __grid_constant__ CUtensorMap map_vb,
                         const __grid_constant__ CUtensorMap map_hb, int n, int nb, float scale,
                         const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
                         int max_sel, int ucap, const int32_t* __restrict__ plan,
                         void* __restrict__ out, int out_bf16, int32_t* status) {
  using SM = Smem<D>;
  constexpr int TILE_BYTES = SM::TILE_BYTES;
  constexpr int PANELS = D / 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::MISC + 4);
  int* s_nu = reinterpret_cast<int*>(smem + SM::MISC + 8);  // [2] union sizes
  const int nwords = ceil_div(nb, 32);
  uint32_t* qmask = reinterpret_cast<uint32_t*>(smem + SM::MASK);  // [4][nwords] per query block
  uint32_t* umask = qmask + 4 * nwords;                              // [2][nwords] per query tile
  uint16_t* ulist = reinterpret_cast<uint16_t*>(umask + 2 * nwords);  // [2][ucap], ascending

  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int h = blockIdx.y;
  const int n_chunks = ceil_div(nb, 128);
  // this CTA's four query blocks: block x holds rows 64 (x & 1) to 64 (x & 1)
  // + 63 of query tile x >> 1; nb stands for no block (rows read as zero,
  // nothing written)
  int qblk[4];
  {
    const int32_t* pr = plan + (static_cast<size_t>(h) * gridDim.x + blockIdx.x) * 4;
    bool bad = false;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      qblk[x] = pr[x];
      bad |= qblk[x] < 0 || qblk[x] > nb;
    }
    if (bad) {
      if (tid == 0) report(status, PISA_ERR_DEVICE_CHECK);
#pragma unroll
      for (int x = 0; x < 4; ++x) qblk[x] = nb;
    }
  }

  // ---- set-up: barriers, TMEM, route bitmasks, union of the critical sets ----
  if (tid == 0) {
    *abort = 0;
    tc::mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&bars[B_KFULL + s], 1);
      tc::mbar_init(&bars[B_KEMPTY + s], 1);
      tc::mbar_init(&bars[B_VFULL + s], 1);
      tc::mbar_init(&bars[B_VEMPTY + s], 1);
    }
    for (int w = 0; w < TILES; ++w) {
      tc::mbar_init(&bars[B_SFULL + w], 1);
      tc::mbar_init(&bars[B_PFULL + 2 * w], TILE_M);
      tc::mbar_init(&bars[B_PFULL + 2 * w + 1], TILE_M);
      tc::mbar_init(&bars[B_OFULL + w], 1);
    }
    tc::mbar_init(&bars[B_DRAIN], 1);
    tc::fence_barrier_init();
  }
  if (warp == WARP_MMA) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  for (int e = tid; e < 6 * nwords; e += NUM_THREADS) qmask[e] = 0u;
  __syncthreads();
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int qb = qblk[x];
    if (qb >= nb) continue;
    const int c = min(cnt[static_cast<size_t>(h) * nb + qb], max_sel);
    const int32_t* lst = idx + (static_cast<size_t>(h) * nb + qb) * max_sel;
    for (int e = tid; e < c; e += NUM_THREADS) {
      const int j = lst[e];
      if (j >= 0 && j < nb) {
        atomicOr(&qmask[x * nwords + j / 32], 1u << (j % 32));
        atomicOr(&umask[(x >> 1) * nwords + j / 32], 1u << (j % 32));
      } else {
        report(status, PISA_ERR_DEVICE_CHECK);
      }
    }
  }
  __syncthreads();
  if (warp < TILES) {
    // warp w compacts the union of query tile w into an ascending list
    const uint32_t* um = umask + warp * nwords;
    uint16_t* ul = ulist + warp * ucap;
    int base = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int wd = w0 + lane;
      const uint32_t bits = (wd < nwords) ? um[wd] : 0u;
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = base + incl - c;
      uint32_t b = bits;
      while (b) {
        const int t = __ffs(b) - 1;
        b &= b - 1;
        if (pos < ucap) ul[pos] = static_cast<uint16_t>(wd * 32 + t);
        ++pos;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_nu[warp] = min(base, ucap);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int te_w[TILES];  // exact tiles of each query tile
  for (int w = 0; w < TILES; ++w) te_w[w] = ceil_div(s_nu[w], 2);
  const int s_ex = max(te_w[0], te_w[1]);  // exact steps
  const int n_steps = s_ex + n_chunks;

  unsigned char* sQ = smem + SM::Q;
  unsigned char* sK = smem + SM::K;
  unsigned char* sV = smem + SM::V;

  if (warp == WARP_TMA) {
    // =========================== TMA producers ===============================
    if (lane < 2) {
      const bool is_k = lane == 0;
      unsigned char* ring = is_k ? sK : sV;
      uint64_t* full = &bars[is_k ? B_KFULL : B_VFULL];
      uint64_t* empty = &bars[is_k ? B_KEMPTY : B_VEMPTY];
      const CUtensorMap* gmap = is_k ? &map_k : &map_v;
      const CUtensorMap* cmap = is_k ? &map_kb : &map_vb;
      tc::prefetch_tmap(gmap);
      tc::prefetch_tmap(cmap);
      if (is_k) {
        tc::prefetch_tmap(&map_q);
        tc::mbar_arrive_expect_tx(&bars[B_Q], TILES * TILE_BYTES);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          for (int p = 0; p < PANELS; ++p)
            tc::tma_load_3d(sQ + (x >> 1) * TILE_BYTES + p * PANEL + (x & 1) * HALF_PANEL, &map_q,
                            64 * p, qblk[x] * kBlock, h, &bars[B_Q]);
      } else {
        tc::prefetch_tmap(&map_hb);
      }
      // the load sequence, identical on both rings and in the MMA issuer:
      // exact step s: tile s of query tile 0 (if any), then of query tile 1;
      // centroid chunk c: hi, lo; and on the V ring Hbar hi, lo at the end.
      int issued = 0;
      bool go = true;
      auto next = [&](auto&& issue) {
        if (!go) return;
        const int l = issued;
        const int s = l % STAGES;
        const uint32_t use = l / STAGES;
        if (l >= STAGES && !wait_or_abort(&empty[s], (use - 1) & 1, abort, status)) {
          go = false;
          return;
        }
        tc::mbar_arrive_expect_tx(&full[s], TILE_BYTES);
        issue(ring + s * TILE_BYTES, &full[s]);
        issued = l + 1;
      };
      for (int st = 0; st < s_ex && go; ++st) {
        for (int w = 0; w < TILES; ++w) {
          if (st >= te_w[w]) continue;
          const uint16_t* ul = ulist + w * ucap;
          const int ja = ul[2 * st];
          const int jb = (2 * st + 1 < s_nu[w]) ? ul[2 * st + 1] : ja;
          next([&](unsigned char* dst, uint64_t* bar) {
            for (int p = 0; p < PANELS; ++p) {
              tc::tma_load_3d(dst + p * PANEL, gmap, 64 * p, ja * kBlock, h, bar);
              tc::tma_load_3d(dst + p * PANEL + HALF_PANEL, gmap, 64 * p, jb * kBlock, h, bar);
            }
          });
        }
      }
      for (int c = 0; c < n_chunks && go; ++c)
        for (int part = 0; part < 2; ++part)
          next([&](unsigned char* dst, uint64_t* bar) {
            for (int p = 0; p < PANELS; ++p)
              tc::tma_load_3d(dst + p * PANEL, cmap, 64 * p, 128 * c, 2 * h + part, bar);
          });
      if (!is_k)
        for (int part = 0; part < 2; ++part)
          next([&](unsigned char* dst, uint64_t* bar) {
            for (int p = 0; p < PANELS; ++p)  // rows past D of a d = 64 Hbar read as 0
              tc::tma_load_3d(dst + p * PANEL, &map_hb, 64 * p, 0, 2 * h + part, bar);
          });
      if (*abort) {
        int zero = 0;
        for (int l = max(0, issued - STAGES); l < issued; ++l)
          tc::mbar_wait(&full[l % STAGES], (l / STAGES) & 1, &zero, WAIT_LIMIT);
        if (is_k) tc::mbar_wait(&bars[B_Q], 0, &zero, WAIT_LIMIT);
      }
    }
  } else if (warp == WARP_MMA) {
    // =========================== MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(TILE_M, 128, false);
      constexpr uint32_t IDESC_PV = tc::idesc_bf16_f32(TILE_M, D, true);
      const uint32_t q0 = tc::smem_u32(sQ), k0 = tc::smem_u32(sK), v0 = tc::smem_u32(sV);
      // Descriptors of the Q tiles and ring stages, built once: a K-step then
      // only adds its byte offset / 16 to the start-address field (shared
      // addresses stay below 2^18, so the 14-bit field never carries).
      const uint64_t dq0 = tc::smem_desc_sw128(q0, 16, 1024);
      const uint64_t dq1 = tc::smem_desc_sw128(q0 + TILE_BYTES, 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(k0, 16, 1024);
      const uint64_t dk1 = tc::smem_desc_sw128(k0 + TILE_BYTES, 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(v0, PANEL, 1024);
      const uint64_t dv1 = tc::smem_desc_sw128(v0 + TILE_BYTES, PANEL, 1024);
      static_assert(STAGES == 2, "one descriptor per ring stage");
      // S_w (+)= Q_w B^T with B from K stage s (D / 16 K-steps of 16 channels)
      auto mma_s = [&](int w, int s, bool acc) {
        tc::mma_ss_ksteps<D / 16>(tmem + w * 128, w ? dq1 : dq0, s ? dk1 : dk0, IDESC_S,
                                  acc ? 1u : 0u);
      };
      // D (+)= P_w B for keys of one half (4 K-steps) with B from V stage s
      auto mma_pv_half = [&](uint32_t d_tmem, int w, int s, int half, bool acc) {
        tc::mma_ts_k4(d_tmem, tmem + w * 128 + 32 * half, (s ? dv1 : dv0) + 512 * half, IDESC_PV,
                      (acc || half > 0) ? 1u : 0u);
      };
      auto wait_k = [&](int l) {
        const bool r = wait_or_abort(&bars[B_KFULL + l % STAGES], (l / STAGES) & 1, abort, status);
        tc::tc_fence_after();
        return r;
      };
      auto wait_v = [&](int l) {
        const bool r = wait_or_abort(&bars[B_VFULL + l % STAGES], (l / STAGES) & 1, abort, status);
        tc::tc_fence_after();
        return r;
      };
      // One tile of query tile w: its first K and V load indices on the rings,
      // the tile's index u in w's own sequence, and whether it is a centroid
      // tile (two loads: hi and lo).
      struct Rec {
        int k, v, u;
        bool two;
      };
      auto wait_loads = [&](bool is_k, int l, bool two) {
        if (!(is_k ? wait_k(l) : wait_v(l))) return false;
        return !two || (is_k ? wait_k(l + 1) : wait_v(l + 1));
      };
      auto release = [&](int base, int l, bool two) {
        tc::mma_commit(&bars[base + l % STAGES]);
        if (two) tc::mma_commit(&bars[base + (l + 1) % STAGES]);
      };
      auto issue_s = [&](int w, const Rec& rc) {
        mma_s(w, rc.k % STAGES, false);
        if (rc.two) mma_s(w, (rc.k + 1) % STAGES, true);  // + Kbar_lo
        tc::mma_commit(&bars[B_SFULL + w]);
      };
      // O_w += P_w V (two halves, each gated by its P barrier)
      auto issue_pv = [&](int w, const Rec& rc) -> bool {
        for (int half = 0; half < 2; ++half) {
          if (!wait_or_abort(&bars[B_PFULL + 2 * w + half], rc.u & 1, abort, status)) return false;
          tc::tc_fence_after();
          mma_pv_half(tmem + 256 + w * 128, w, rc.v % STAGES, half, rc.u > 0);
          if (rc.two) mma_pv_half(tmem + 256 + w * 128, w, (rc.v + 1) % STAGES, half, true);
        }
        return true;
      };

      // Step order (same as the block-wise kernel): S0, P V of query tile 1's
      // previous tile, S1, P V of query tile 0. Each S_w is thus issued after
      // the P V that last read its TMEM columns.
      bool ok = wait_or_abort(&bars[B_Q], 0, abort, status);
      // While both query tiles stream exact tiles, step st puts tile 0's K and
      // V in stage 0 and tile 1's in stage 1 (load 2 st and 2 st + 1 on each
      // ring), with phase st & 1: the same products, commits and waits as the
      // general loop below, without its per-step bookkeeping.
      const int m_both = min(te_w[0], te_w[1]);
      int st = 0;
      for (; ok && st < m_both; ++st) {
        const uint32_t ph = st & 1;
        if (!(ok = wait_or_abort(&bars[B_KFULL + 0], ph, abort, status))) break;
        tc::tc_fence_after();
        mma_s(0, 0, false);
        tc::mma_commit(&bars[B_SFULL + 0]);
        tc::mma_commit(&bars[B_KEMPTY + 0]);
        if (st > 0) {
          if (!(ok = wait_or_abort(&bars[B_VFULL + 1], ph ^ 1u, abort, status))) break;
          tc::tc_fence_after();
          if (!(ok = issue_pv(1, Rec{2 * st - 1, 2 * st - 1, st - 1, false}))) break;
          tc::mma_commit(&bars[B_VEMPTY + 1]);
        }
        if (!(ok = wait_or_abort(&bars[B_KFULL + 1], ph, abort, status))) break;
        tc::tc_fence_after();
        mma_s(1, 1, false);
        tc::mma_commit(&bars[B_SFULL + 1]);
        tc::mma_commit(&bars[B_KEMPTY + 1]);
        if (!(ok = wait_or_abort(&bars[B_VFULL + 0], ph, abort, status))) break;
        tc::tc_fence_after();
        if (!(ok = issue_pv(0, Rec{2 * st, 2 * st, st, false}))) break;
        tc::mma_commit(&bars[B_VEMPTY + 0]);
      }
      int kcnt = 2 * m_both, vcnt = 2 * m_both;
      int uw[TILES] = {m_both, m_both};
      Rec pend{2 * m_both - 1, 2 * m_both - 1, m_both - 1, false};
      bool has_pend = m_both > 0;
      for (; ok && st < n_steps; ++st) {
        const bool cen = st >= s_ex;
        Rec rc[TILES];
        bool has[TILES];
        for (int w = 0; w < TILES; ++w) {
          has[w] = cen || st < te_w[w];
          if (has[w]) rc[w] = Rec{cen ? kcnt : kcnt++, cen ? vcnt : vcnt++, uw[w], cen};
          uw[w] += has[w] ? 1 : 0;
        }
        if (cen) {
          kcnt += 2;
          vcnt += 2;
        }
        // An exact tile's K stage is freed as soon as its own S product is
        // done; a centroid pair (read by both S products) after S1.
        if (has[0]) {
          if (!(ok = wait_loads(true, rc[0].k, rc[0].two))) break;
          issue_s(0, rc[0]);
          if (!cen) release(B_KEMPTY, rc[0].k, false);
        }
        if (has_pend) {
          if (!(ok = wait_loads(false, pend.v, pend.two))) break;
          if (!(ok = issue_pv(1, pend))) break;
          release(B_VEMPTY, pend.v, pend.two);
          has_pend = false;
        }
        if (has[1]) {
          if (!(ok = wait_loads(true, rc[1].k, rc[1].two))) break;
          issue_s(1, rc[1]);
          release(B_KEMPTY, rc[1].k, cen);
        }
        if (has[0]) {
          if (!(ok = wait_loads(false, rc[0].v, rc[0].two))) break;
          if (!(ok = issue_pv(0, rc[0]))) break;
          if (!cen) release(B_VEMPTY, rc[0].v, false);  // a centroid pair waits for tile 1
        }
        if (has[1]) {
          pend = rc[1];
          has_pend = true;
        }
      }
      if (ok && has_pend) {
        ok = wait_loads(false, pend.v, pend.two) && issue_pv(1, pend);
        if (ok) release(B_VEMPTY, pend.v, pend.two);
      }
      if (ok) {
        // first order: Q_w (Hbar_hi + Hbar_lo) into the S columns of tile w
        const int l = vcnt;
        ok = wait_v(l) && wait_v(l + 1);
        if (ok) {
          for (int w = 0; w < TILES; ++w) {
            const uint32_t qa = q0 + w * TILE_BYTES;
            for (int part = 0; part < 2; ++part) {
              const uint32_t ha = v0 + ((l + part) % STAGES) * TILE_BYTES;
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks >> 2) * PANEL + (ks & 3) * 32;
                tc::mma_ss(tmem + w * 128, tc::smem_desc_sw128(qa + off, 16, 1024),
                           tc::smem_desc_sw128(ha + ks * 2048, PANEL, 1024), IDESC_PV,
                           (part > 0 || ks > 0) ? 1u : 0u);
              }
            }
            tc::mma_commit(&bars[B_OFULL + w]);
          }
        }
      }
      int zero = 0;
      tc::mma_commit(&bars[B_DRAIN]);
      tc::mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_LIMIT);
    }
  } else {
    // ====================== softmax / epilogue warpgroups =====================
    const int w = warp / 4;
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const int x = 2 * w + (wq >> 1);
    const int my_qb = (x & 2) ? ((x & 1) ? qblk[3] : qblk[2]) : ((x & 1) ? qblk[1] : qblk[0]);
    const uint32_t* mask = qmask + x * nwords;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + w * 128 + lane_off;
    const uint32_t tO = tmem + 256 + w * 128 + lane_off;
    const float sl2 = scale * 1.4426950408889634f;
    const int last_n = n - (nb - 1) * kBlock;  // keys of the last block
    const int te = w ? te_w[1] : te_w[0];  // exact tiles and union size of tile w
    const int nu = s_nu[w];
    const uint16_t* ul = ulist + w * ucap;
    const int T = te + n_chunks;
    float m_run = -INFINITY, l_run = 0.f, tail = 0.f;
    bool ok = true;
    // Online-softmax shift for a tile whose row maximum is mt2 (log2 units):
    // the first contribution of a row sets it (O, l and tail are still 0);
    // later it moves only when mt2 exceeds it by more than 2^LAZY. Rows with
    // no contribution yet keep m_run = -inf and P = 0, which is exact even
    // though O holds garbage before the first accumulating P V.
    auto shift = [&](float mt2) {
      if (mt2 != -INFINITY && m_run == -INFINITY) m_run = mt2;
      const bool need = mt2 != -INFINITY && mt2 > m_run + LAZY;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2_approx(m_run - mt2) : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 8; ++c) {
          uint32_t ov[8];
          tc::tmem_ld8(tO + 8 * c, ov);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          tc::tmem_st8(tO + 8 * c, ov);
        }
        if (need) {
          l_run *= f;
          tail *= f;
          m_run = mt2;
        }
      }
    };

    // tcgen05.ld/st are warp-collective: every branch around them is
    // warp-uniform (a warp's 32 rows lie in one query block).
    for (int t = 0; t < T; ++t) {
      ok = wait_or_abort(&bars[B_SFULL + w], t & 1, abort, status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint64_t sl2x2 = f2f(sl2, sl2);
      if (t < te) {
        // ---- exact tile: halves are blocks ul[2t], ul[2t+1]; a half whose
        // block is not critical for this query block (or the repeated block of
        // an odd union) gets P = 0
        uint32_t sv[4][32];
        tc::tmem_ld32(tS, sv[0]);
        tc::tmem_ld32(tS + 32, sv[1]);
        tc::tmem_wait_ld();
        after_wait(sv[0]);
        after_wait(sv[1]);
        tc::tmem_ld32(tS + 64, sv[2]);
        tc::tmem_ld32(tS + 96, sv[3]);
        float mt = -INFINITY;
        bool ex[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int u = 2 * t + hh;
          const int j = (u < nu) ? ul[u] : 0;
          ex[hh] = u < nu && ((mask[j >> 5] >> (j & 31)) & 1u);
          if (hh == 1) {
            tc::tmem_wait_ld();
            after_wait(sv[2]);
            after_wait(sv[3]);
          }
          if (ex[hh]) {
            if (j == nb - 1 && last_n < kBlock) mask_tail(sv[2 * hh], sv[2 * hh + 1], last_n);
            mt = fmaxf(mt, row_max64(sv[2 * hh], sv[2 * hh + 1]));
          }
        }
        shift(mt * sl2);
        const uint64_t nm2 = f2f(-m_run, -m_run);
        // The tile's largest exact weight enters P V rounded to bf16. Under the
        // lazy shift it can be up to 2^20, and in a row dominated by one key
        // its rounding (up to 2^-9 of it) would show in the output; adding
        // that rounding to the denominator keeps numerator and denominator
        // consistent for the dominant key (the other keys' roundings are
        // small and random). Same operations as the loop below, so the same
        // value.
        if (mt != -INFINITY) {
          const float pm = ex2_approx(fmaf(mt, sl2, -m_run));
          float r0, r1;
          unf2(unpack_bf16x2(pack_bf16(pm, 0.f)), r0, r1);
          l_run += r0 - pm;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (ex[hh]) {
            uint64_t ls[2] = {0ull, 0ull};
#pragma unroll
            for (int q32 = 0; q32 < 2; ++q32) {
              const uint32_t(&src)[32] = sv[2 * hh + q32];
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float z0, z1;
                unf2(fma2(f2(src[2 * e], src[2 * e + 1]), sl2x2, nm2), z0, z1);
                const float p0 = ex2_approx(z0), p1 = ex2_approx(z1);
                ls[e & 1] = add2(ls[e & 1], f2f(p0, p1));
                pk[e] = pack_bf16(p0, p1);
              }
              tc::tmem_st16(tS + 32 * hh + 16 * q32, pk);
            }
            float l0, l1;
            unf2(add2(ls[0], ls[1]), l0, l1);
            l_run += l0 + l1;
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
            tc::tmem_st16(tS + 32 * hh, pk);
            tc::tmem_st16(tS + 32 * hh + 16, pk);
          }
          tc::tmem_wait_st();
          tc::tc_fence_before();
          tc::mbar_arrive(&bars[B_PFULL + 2 * w + hh]);
        }
      } else {
        // ---- centroid tile (a few per row), column c <-> block j0 + c: one
        // 32-column group at a time, read from TMEM, in rolled loops that keep
        // this rare path's code small
        const int j0 = 128 * (t - te);
        float mt = -INFINITY;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t x[32];
          tc::tmem_ld32(tS + 32 * g, x);
          tc::tmem_wait_ld();
          after_wait(x);
          const uint32_t cm = centroid_cols(mask, j0 + 32 * g, nb);
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m4[i & 3] = fmaxf(m4[i & 3], ((cm >> i) & 1u) ? __uint_as_float(x[i]) : -INFINITY);
          mt = max3(mt, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        shift(mt * sl2);
        const uint64_t nm2 = f2f(-m_run, -m_run);
        // P = alpha on the counted columns; mass n_j alpha (n_j = 64 except
        // for a partial last block). P of group g (16 packed columns) lands on
        // S columns [16 g, 16 g + 16), already read for every g.
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t x[32];
          tc::tmem_ld32(tS + 32 * g, x);
          tc::tmem_wait_ld();
          after_wait(x);
          const uint32_t cm = centroid_cols(mask, j0 + 32 * g, nb);
          const int cl = (nb - 1) - (j0 + 32 * g);  // column of the last block
          uint64_t ts2 = 0ull;
          float plast = 0.f;
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float z0, z1;
            unf2(fma2(f2(x[2 * e], x[2 * e + 1]), sl2x2, nm2), z0, z1);
            float p0 = ((cm >> (2 * e)) & 1u) ? ex2_approx(z0) : 0.f;
            float p1 = ((cm >> (2 * e + 1)) & 1u) ? ex2_approx(z1) : 0.f;
            // the centroid weights as rounded for the tensor cores: the mass and
            // the first-order weight use the same numbers
            pk[e] = pack_bf16(p0, p1);
            const uint64_t pr = unpack_bf16x2(pk[e]);
            unf2(pr, p0, p1);
            plast = (cl == 2 * e) ? p0 : ((cl == 2 * e + 1) ? p1 : plast);
            ts2 = add2(ts2, pr);
          }
          tc::tmem_st16(tS + 16 * g, pk);
          float t0, t1;
          unf2(ts2, t0, t1);
          const float ts = t0 + t1;
          l_run = fmaf(static_cast<float>(kBlock), ts,
                       fmaf(static_cast<float>(last_n - kBlock), plast, l_run));
          tail += ts;
          if (g & 1) {
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&bars[B_PFULL + 2 * w + (g >> 1)]);
          }
        }
      }
    }

    // ---- epilogue: o = (O + s tail Q Hbar) / l --------------------------------
    if (ok) ok = wait_or_abort(&bars[B_OFULL + w], 0, abort, status);
    if (__all_sync(0xffffffffu, ok)) {
      tc::tc_fence_after();
      const int row = my_qb * kBlock + (r & (kBlock - 1));
      const float inv = 1.f / l_run;
      const float st = scale * tail;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32], hv[32];
        tc::tmem_ld32(tO + 32 * c, ov);
        tc::tmem_ld32(tS + 32 * c, hv);
        tc::tmem_wait_ld();
        after_wait(ov);
        after_wait(hv);
        float res[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          res[e] = fmaf(st, __uint_as_float(hv[e]), __uint_as_float(ov[e])) * inv;
        if (my_qb < nb && row < n) {
          const size_t base = (static_cast<size_t>(h) * n + row) * D + 32 * c;
          if (out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + base);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 u;
              u.x = pack_bf16(res[8 * e + 0], res[8 * e + 1]);
              u.y = pack_bf16(res[8 * e + 2], res[8 * e + 3]);
              u.z = pack_bf16(res[8 * e + 4], res[8 * e + 5]);
              u.w = pack_bf16(res[8 * e + 6], res[8 * e + 7]);
              dst[e] = u;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(res[4 * e], res[4 * e + 1], res[4 * e + 2], res[4 * e + 3]);
          }
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// fp32 -> bf16 hi + lo (lo = bf16(x - hi)) for the centroid and Hbar operands
__global__ void split_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                  int heads, size_t per_head) {
  const size_t total = static_cast<size_t>(heads) * per_head;
  for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t hh = e / per_head, o = e % per_head;
    const float x = src[e];
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    dst[(2 * hh) * per_head + o] = hi;
    dst[(2 * hh + 1) * per_head + o] = lo;
  }
}

bool map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {64, b1, 1};
  return make_tmap_bf16(m, base, 3, dims, strides, box);
}

}  // namespace

size_t forward_hybrid_tc_operand_bytes(int heads, int n, int d) {
  const size_t nb = static_cast<size_t>(ceil_div(n, kBlock));
  return (2 * 2 * static_cast<size_t>(heads) * nb * d + 2 * static_cast<size_t>(heads) * d * d) *
         sizeof(__nv_bfloat16);
}

size_t forward_hybrid_tc_plan_bytes(int heads, int n) {
  return static_cast<size_t>(heads) * 4 * ceil_div(n, CTA_ROWS) * sizeof(int32_t);
}

size_t forward_hybrid_tc_workspace(int heads, int n, int d) {
  const size_t ops = (forward_hybrid_tc_operand_bytes(heads, n, d) + 255) & ~static_cast<size_t>(255);
  return ops + forward_hybrid_tc_plan_bytes(heads, n);
}

namespace {

template <int D>
int launch_hybrid(const void* q, const void* k, const void* v, int heads, int n, float scale,
                  const float* kbar, const float* vsum, const float* hbar, const int32_t* idx,
                  const int32_t* cnt, int max_sel, void* out, int out_bf16, void* workspace,
                  int32_t* plan, int32_t* dev_status, cudaStream_t stream) {
  const int nb = ceil_div(n, kBlock);
  if (ceil_div(nb, 2) > kHybridPlanMaxTiles) return PISA_ERR_UNSUPPORTED;
  __nv_bfloat16* kb2 = static_cast<__nv_bfloat16*>(workspace);
  __nv_bfloat16* vb2 = kb2 + 2 * static_cast<size_t>(heads) * nb * D;
  __nv_bfloat16* hb2 = vb2 + 2 * static_cast<size_t>(heads) * nb * D;
  const int threads = 256;
  auto split = [&](const float* src, __nv_bfloat16* dst, size_t per_head) -> int {
    const size_t total = static_cast<size_t>(heads) * per_head;
    const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 4096));
    split_bf16_kernel<<<blocks, threads, 0, stream>>>(src, dst, heads, per_head);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  int rc;
  if ((rc = split(kbar, kb2, static_cast<size_t>(nb) * D)) != PISA_OK) return rc;
  if ((rc = split(vsum, vb2, static_cast<size_t>(nb) * D)) != PISA_OK) return rc;
  if ((rc = split(hbar, hb2, static_cast<size_t>(D) * D)) != PISA_OK) return rc;
  if ((rc = launch_hybrid_plan(idx, cnt, heads, nb, max_sel, plan, stream)) != PISA_OK) return rc;

  CUtensorMap mq, mk, mv, mkb, mvb, mhb;
  const uint64_t H = heads, N = n, NB = nb;
  if (!map3(&mq, q, D, N, H, 64) || !map3(&mk, k, D, N, H, 64) || !map3(&mv, v, D, N, H, 64) ||
      !map3(&mkb, kb2, D, NB, 2 * H, 128) || !map3(&mvb, vb2, D, NB, 2 * H, 128) ||
      !map3(&mhb, hb2, D, D, 2 * H, 128))
    return PISA_ERR_CUDA;
  const int nwords = ceil_div(nb, 32);
  const int ucap = static_cast<int>(std::min<long long>(nb, 2LL * max_sel));  // union of 2 sets
  const long long smem_ll = Smem<D>::MASK + 6LL * nwords * 4 + 2LL * 2 * ucap + 1024;
  if (smem_ll > 232448) return PISA_ERR_UNSUPPORTED;  // very large dense routes
  const int smem = static_cast<int>(smem_ll);
  PISA_CUDA_TRY(cudaFuncSetAttribute(forward_hybrid_tc_kernel<D>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  dim3 grid(ceil_div(n, CTA_ROWS), heads);  // = ceil(n_tiles / 2) pairs of query tiles
  forward_hybrid_tc_kernel<D><<<grid, NUM_THREADS, smem, stream>>>(mq, mk, mv, mkb, mvb, mhb, n, nb,
                                                                scale, idx, cnt, max_sel, ucap,
                                                                plan, out, out_bf16, dev_status);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}

}  // namespace

int launch_forward_hybrid_tc(const void* q, const void* k, const void* v, int heads, int n, int d,
                             float scale, const float* kbar, const float* vsum, const float* hbar,
                             const int32_t* idx, const int32_t* cnt, int max_sel, void* out,
                             int out_bf16, void* workspace, int32_t* plan, int32_t* dev_status,
                             cudaStream_t stream) {
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  return d == 128 ? launch_hybrid<128>(q, k, v, heads, n, scale, kbar, vsum, hbar, idx, cnt,
                                       max_sel, out, out_bf16, workspace, plan, dev_status, stream)
                  : launch_hybrid<64>(q, k, v, heads, n, scale, kbar, vsum, hbar, idx, cnt,
                                      max_sel, out, out_bf16, workspace, plan, dev_status, stream);
}

}  // namespace pisa
