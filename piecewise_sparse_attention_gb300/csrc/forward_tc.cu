// Piecewise forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// for bf16 inputs with head dim 128 or 64 (template parameter D: a [128][D]
// tile is D / 64 swizzled panels; O uses D of its 128 TMEM columns).
//
// "PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
// Transformers", Section 3.2, Eq. (3)-(6). For a key block j outside the
// critical set S_i, the block-wise first-order terms
//     n_j e^{a}  (denominator)   and   e^{a} (Vhat_j + q' H_j)  (numerator),
// a = q'.kbar_j, are evaluated in their token-level form
//     e^{a} sum_n (1 + q'.k_{j,n} - a) v_{j,n},   a = mean_n q'.k_{j,n},
// which is the same number (kbar_j is the mean key and H_j = sum_n (k_{j,n} -
// kbar_j)^T v_{j,n}). The whole forward then has the shape of one dense
// attention pass: S = Q K^T for every key block, an element-wise weight P
// (exp for critical blocks, one fused multiply-add for approximated ones) and
// O += P V, all on the tensor cores; only the element-wise step differs per
// (query block, key block) pair.
//
// CTA = 256 query rows of one head (two 128-row tiles), 10 warps:
//   warps 0-3  softmax/epilogue for tile 0 (TMEM lanes 0-127, S0/P0, O0)
//   warps 4-7  softmax/epilogue for tile 1 (S1/P1, O1)
//   warp  8    TMA producers: lane 0 Q once then K, lane 1 V (128-key tiles,
//              2-stage ring each)
//   warp  9    TMEM allocator and single-thread tcgen05.mma issuer
// TMEM columns: S0 [0,128) (P0 aliases [0,64) as packed bf16), S1 [128,256),
// O0 [256,384), O1 [384,512).
// MMA issue order per key tile t: S0_t, PV1_{t-1}, S1_t, PV0_t. Every S_t of a
// tile is issued after the PV that last read the same TMEM columns, and the
// commit that publishes S_t also covers that PV, so a softmax warpgroup that
// sees S_t may rescale its O accumulator in place.
// Online softmax with a lazy shift: the running maximum is only moved when a
// tile exceeds it by more than 2^20 (weights up to 2^20 and sums over at most
// 2^20 keys stay far inside the bf16/float32 range), which skips almost every
// O rescale.
// Every wait is bounded; on expiry the kernel stores PISA_ERR_TIMEOUT in the
// status word, drains its in-flight copies and MMAs, frees TMEM and returns.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "rowops.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace pisa {
namespace {

constexpr int TILE_M = 128;               // query rows per tile
constexpr int TILES = 2;                  // query tiles per CTA
constexpr int CTA_ROWS = TILE_M * TILES;  // 256
constexpr int TILE_N = 128;               // keys per key tile (two blocks)
constexpr int STAGES = 2;
constexpr int PANEL = 128 * 128;          // bytes of a [128 rows][64 bf16] panel
constexpr int NUM_THREADS = 320;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr long long WAIT_LIMIT = 2000000000LL;  // ~1 s of SM clock per wait
constexpr float LAZY = 20.0f;                   // log2 headroom before a rescale

// byte offsets inside the 1024-aligned dynamic shared memory; a [128 rows][D]
// tile is D / 64 panels
template <int D>
struct Smem {
  static constexpr int TILE_BYTES = D / 64 * PANEL;
  static constexpr int Q = 0;                              // TILES x TILE_BYTES
  static constexpr int K = Q + TILES * TILE_BYTES;         // STAGES x TILE_BYTES
  static constexpr int V = K + STAGES * TILE_BYTES;        // STAGES x TILE_BYTES
  static constexpr int BAR = V + STAGES * TILE_BYTES;      // mbarriers
  static constexpr int NBAR = 20;
  static constexpr int MISC = BAR + NBAR * 8;              // tmem slot, abort flag
  static constexpr int MASK = MISC + 64;                   // route bitmasks
};

// barrier indices
enum {
  B_Q = 0,
  B_KFULL = 1,   // +stage
  B_KEMPTY = 3,  // +stage
  B_VFULL = 5,   // +stage
  B_VEMPTY = 7,  // +stage
  B_SFULL = 9,   // +tile
  B_PFULL = 11,  // +2*tile+half: P of keys [64 half, 64 half + 64) is in TMEM
  B_OFULL = 15,  // +tile
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

// SPREAD: the logit of every approximated block gains w_ij from the
// [heads, nb, nb] matrix `spread` (second-order block mass of the
// Piecewise-Taylor-Attention README); its weights become
// e^{a + w - m}(1 + s (S - a)) and its mass n_j e^{a + w - m}.
template <int D, bool SPREAD>
__global__ void __launch_bounds__(NUM_THREADS, 1)
forward_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                  const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, int n, int nb, float scale,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int max_sel,
                  void* __restrict__ out, int out_bf16, int32_t* status,
                  const float* __restrict__ spread) {
  using SM = Smem<D>;
  constexpr int TILE_BYTES = SM::TILE_BYTES;
  constexpr int PANELS = D / 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::MISC + 4);
  uint32_t* qmask = reinterpret_cast<uint32_t*>(smem + SM::MASK);

  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int h = blockIdx.y;
  const int row_base = blockIdx.x * CTA_ROWS;       // first query row of the CTA
  const int qb_base = row_base / kBlock;             // first query block
  const int nwords = ceil_div(nb, 32);
  const int T = ceil_div(nb, 2);                     // key tiles
  // Step t works on key tile (t0 + t) mod T: the CTA starts at its diagonal,
  // so the first tile's maximum (in peaked rows the row's largest logit)
  // sets the running shift and the dominant weights come out near 1.
  const int t0 = min(T - 1, max(0, qb_base - 1) / 2);
  auto tile_of = [&](int t) { return t0 + t < T ? t0 + t : t0 + t - T; };

  // ---- set-up: barriers, TMEM, route bitmasks --------------------------------
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
  for (int e = tid; e < 4 * nwords; e += NUM_THREADS) qmask[e] = 0u;
  __syncthreads();
  for (int x = 0; x < 4; ++x) {
    const int qb = qb_base + x;
    if (qb >= nb) break;
    const int c = min(cnt[static_cast<size_t>(h) * nb + qb], max_sel);
    const int32_t* lst = idx + (static_cast<size_t>(h) * nb + qb) * max_sel;
    for (int e = tid; e < c; e += NUM_THREADS) {
      const int j = lst[e];
      if (j >= 0 && j < nb) atomicOr(&qmask[x * nwords + j / 32], 1u << (j % 32));
      else report(status, PISA_ERR_DEVICE_CHECK);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  unsigned char* sQ = smem + SM::Q;
  unsigned char* sK = smem + SM::K;
  unsigned char* sV = smem + SM::V;

  if (warp == WARP_TMA) {
    // =========================== TMA producers ===============================
    // lane 0 streams Q once and then K, lane 1 streams V: the two rings are
    // released at different points of the MMA order (K after both S MMAs, V
    // after both P V MMAs), so neither stream waits behind the other.
    if (lane < 2) {
      const bool is_k = lane == 0;
      const CUtensorMap* map = is_k ? &map_k : &map_v;
      unsigned char* ring = is_k ? sK : sV;
      uint64_t* full = &bars[is_k ? B_KFULL : B_VFULL];
      uint64_t* empty = &bars[is_k ? B_KEMPTY : B_VEMPTY];
      tc::prefetch_tmap(map);
      if (is_k) {
        tc::prefetch_tmap(&map_q);
        tc::mbar_arrive_expect_tx(&bars[B_Q], TILES * TILE_BYTES);
        for (int w = 0; w < TILES; ++w)
          for (int p = 0; p < PANELS; ++p)
            tc::tma_load_3d(sQ + w * TILE_BYTES + p * PANEL, &map_q, 64 * p,
                            row_base + w * TILE_M, h, &bars[B_Q]);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t use = t / STAGES;
        if (t >= STAGES && !wait_or_abort(&empty[s], (use - 1) & 1, abort, status)) break;
        tc::mbar_arrive_expect_tx(&full[s], TILE_BYTES);
        for (int p = 0; p < PANELS; ++p)
          tc::tma_load_3d(ring + s * TILE_BYTES + p * PANEL, map, 64 * p, tile_of(t) * TILE_N, h,
                          &full[s]);
        issued = t + 1;
      }
      if (*abort) {
        // drain: wait (bounded, ignoring the abort flag) for the last copies
        int zero = 0;
        for (int t = max(0, issued - STAGES); t < issued; ++t)
          tc::mbar_wait(&full[t % STAGES], (t / STAGES) & 1, &zero, WAIT_LIMIT);
        if (is_k) tc::mbar_wait(&bars[B_Q], 0, &zero, WAIT_LIMIT);
      }
    }
  } else if (warp == WARP_MMA) {
    // =========================== MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(TILE_M, TILE_N, false);
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
      auto issue_s = [&](int w, int s) {
        tc::mma_ss_ksteps<D / 16>(tmem + w * 128, w ? dq1 : dq0, s ? dk1 : dk0, IDESC_S, 0u);
        tc::mma_commit(&bars[B_SFULL + w]);
      };
      // O_w (+)= P_w V for the 64 keys of one half (4 K-steps of 16)
      auto issue_pv_half = [&](int w, int s, int half, bool acc) {
        tc::mma_ts_k4(tmem + 256 + w * 128, tmem + w * 128 + 32 * half,
                      (s ? dv1 : dv0) + 512 * half, IDESC_PV, (acc || half > 0) ? 1u : 0u);
      };
      // both halves, each issued as soon as its P is ready
      auto issue_pv = [&](int w, int s, int t_of, bool acc) -> bool {
        for (int half = 0; half < 2; ++half) {
          if (!wait_or_abort(&bars[B_PFULL + 2 * w + half], t_of & 1, abort, status)) return false;
          tc::tc_fence_after();
          issue_pv_half(w, s, half, acc);
        }
        return true;
      };
      bool ok = wait_or_abort(&bars[B_Q], 0, abort, status);
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (t / STAGES) & 1;
        if (!(ok = wait_or_abort(&bars[B_KFULL + s], ph, abort, status))) break;
        tc::tc_fence_after();
        issue_s(0, s);
        if (t > 0) {
          const int sp = (t - 1) % STAGES;
          if (!(ok = issue_pv(1, sp, t - 1, t - 1 > 0))) break;
          tc::mma_commit(&bars[B_VEMPTY + sp]);
        }
        issue_s(1, s);
        tc::mma_commit(&bars[B_KEMPTY + s]);
        if (!(ok = wait_or_abort(&bars[B_VFULL + s], ph, abort, status))) break;
        if (!(ok = issue_pv(0, s, t, t > 0))) break;
      }
      if (ok) {
        const int sl = (T - 1) % STAGES;
        ok = issue_pv(1, sl, T - 1, T - 1 > 0);
        if (ok) {
          tc::mma_commit(&bars[B_VEMPTY + sl]);
          tc::mma_commit(&bars[B_OFULL + 0]);
          tc::mma_commit(&bars[B_OFULL + 1]);
        }
      }
      // drain every MMA this thread issued before TMEM is released
      int zero = 0;
      tc::mma_commit(&bars[B_DRAIN]);
      tc::mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_LIMIT);
    }
  } else {
    // ====================== softmax / epilogue warpgroups =====================
    const int w = warp / 4;          // query tile
    const int wq = warp % 4;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // row inside the tile
    const int x = 2 * w + (wq >> 1); // query block slot inside the CTA (0..3)
    const uint32_t* mask = qmask + x * nwords;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + w * 128 + lane_off;
    const uint32_t tO = tmem + 256 + w * 128 + lane_off;
    const float sl2 = scale * 1.4426950408889634f;  // logits in log2 units
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;

    // tcgen05.ld/st are warp-collective: every branch around them below is
    // made warp-uniform (__all_sync / __any_sync) so no lane skips one.
    for (int t = 0; t < T; ++t) {
      const int kt = tile_of(t);  // key tile of this step
      // SPREAD: w for this tile's two key blocks, loaded before the wait for S
      // so that the load's latency overlaps it
      float wpre[2] = {0.f, 0.f};
      if (SPREAD && qb_base + x < nb) {
        const float* wr = spread + (static_cast<size_t>(h) * nb + qb_base + x) * nb;
        if (2 * kt < nb) wpre[0] = __ldg(wr + 2 * kt);
        if (2 * kt + 1 < nb) wpre[1] = __ldg(wr + 2 * kt + 1);
      }
      ok = wait_or_abort(&bars[B_SFULL + w], t & 1, abort, status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      // keys 0-63 first; keys 64-127 are read once half 0 is reduced (issued
      // earlier, their loads held up that reduction)
      uint32_t sv[4][32];
      tc::tmem_ld32(tS, sv[0]);
      tc::tmem_ld32(tS + 32, sv[1]);
      tc::tmem_wait_ld();
      after_wait(sv[0]);
      after_wait(sv[1]);

      // Per 64-key half: number of valid keys (past the end of the sequence the
      // TMA zero-fills K and V, so S = 0 there and P V adds nothing) and
      // whether the block is exact for this warp's query block.
      int nv[2];
      bool ex[2];
      float a[2];
      float ws[2] = {0.f, 0.f};  // SPREAD: w_ij / s (raw logit units)
      float mt = -INFINITY;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = 2 * kt + hh;
        nv[hh] = (j < nb) ? min(kBlock, n - j * kBlock) : 0;
        ex[hh] = nv[hh] > 0 && ((mask[j >> 5] >> (j & 31)) & 1u);
        a[hh] = 0.f;
        if (hh == 1) {
          tc::tmem_ld32(tS + 64, sv[2]);
          tc::tmem_ld32(tS + 96, sv[3]);
          tc::tmem_wait_ld();
          after_wait(sv[2]);
          after_wait(sv[3]);
        }
        if (ex[hh]) {
          if (nv[hh] < kBlock) mask_tail(sv[2 * hh], sv[2 * hh + 1], nv[hh]);  // rare
          mt = fmaxf(mt, row_max64(sv[2 * hh], sv[2 * hh + 1]));
        } else if (nv[hh] > 0) {
          // centroid logit q.kbar_j = mean of the block's logits (zeros past the
          // end add nothing to the sum)
          const float sum = row_sum64(sv[2 * hh], sv[2 * hh + 1]);
          a[hh] = (nv[hh] == kBlock) ? sum * (1.f / kBlock) : sum / static_cast<float>(nv[hh]);
          if (SPREAD) ws[hh] = __fdividef(wpre[hh], scale);  // w in raw logit units
          mt = fmaxf(mt, SPREAD ? a[hh] + ws[hh] : a[hh]);
        }
      }
      const float mt2 = mt * sl2;
      if (t == 0) {
        m_run = mt2;
      } else {
        // move the shift of a row only when its tile maximum exceeds it by more
        // than 2^LAZY; the warp rescales together, other rows by a factor 1
        const bool need = mt2 > m_run + LAZY;
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
            m_run = mt2;
          }
        }
      }
      // P, written back over S as packed bf16 pairs, 32 keys (16 columns) at a
      // time; each half is published on its own barrier so the P V product of
      // keys 0-63 can start while keys 64-127 are still being computed
      const uint64_t nm2 = f2f(-m_run, -m_run);
      const uint64_t sl2x2 = f2f(sl2, sl2);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (ex[hh]) {
          // exact: 2^{S s log2e - m}; masked tail entries are -inf and give 0.
          // The denominator adds the bf16-rounded weights that P V uses.
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
              pk[e] = pack_bf16(p0, p1);
              ls[e & 1] = add2(ls[e & 1], unpack_bf16x2(pk[e]));  // the mass P V sees
            }
            tc::tmem_st16(tS + 32 * hh + 16 * q32, pk);
          }
          float l0, l1;
          unf2(add2(ls[0], ls[1]), l0, l1);
          l_run += l0 + l1;
        } else {
          // first-order expansion around the block's mean logit a:
          // weight c (1 + s (S - a)) = S (c s) + (c - c s a), c = 2^{a s log2e - m};
          // block mass n_j c. An empty half (past the last block) has c = 0.
          const float ae = SPREAD ? a[hh] + ws[hh] : a[hh];
          const float cz = (nv[hh] > 0) ? ex2_approx(fmaf(ae, sl2, -m_run)) : 0.f;
          const float cs = cz * scale;
          const float d0 = fmaf(-cs, a[hh], cz);
          const uint64_t cs2 = f2f(cs, cs), d2 = f2f(d0, d0);
#pragma unroll
          for (int q32 = 0; q32 < 2; ++q32) {
            const uint32_t(&src)[32] = sv[2 * hh + q32];
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float p0, p1;
              unf2(fma2(f2(src[2 * e], src[2 * e + 1]), cs2, d2), p0, p1);
              pk[e] = pack_bf16(p0, p1);
            }
            tc::tmem_st16(tS + 32 * hh + 16 * q32, pk);
          }
          l_run = fmaf(static_cast<float>(nv[hh]), cz, l_run);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[B_PFULL + 2 * w + hh]);
      }
    }

    // ---- epilogue: o = O / l ---------------------------------------------------
    if (ok) ok = wait_or_abort(&bars[B_OFULL + w], 0, abort, status);
    if (__all_sync(0xffffffffu, ok)) {
      tc::tc_fence_after();
      const int row = row_base + w * TILE_M + r;
      const float inv = 1.f / l_run;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tc::tmem_ld32(tO + 32 * c, ov);
        tc::tmem_wait_ld();
        if (row < n) {
          const size_t base = (static_cast<size_t>(h) * n + row) * D + 32 * c;
          if (out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + base);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 u;
              u.x = pack_bf16(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
              u.y = pack_bf16(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
              u.z = pack_bf16(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
              u.w = pack_bf16(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
              dst[e] = u;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(ov[4 * e + 0]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                   __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
          }
        }
      }
    }
  }

  // ---- teardown -----------------------------------------------------------------
  tc::tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

bool make_map(CUtensorMap* m, const void* base, int heads, int n, int d) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(n),
                            static_cast<uint64_t>(heads)};
  const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(n) * d * 2};
  const uint32_t box[3] = {64, 128, 1};
  return make_tmap_bf16(m, base, 3, dims, strides, box);
}

}  // namespace

int launch_forward_tc(const void* q, const void* k, const void* v, int heads, int n, int d,
                      float scale, const int32_t* idx, const int32_t* cnt, int max_sel,
                      void* out, int out_bf16, int32_t* dev_status, cudaStream_t stream,
                      const float* spread) {
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  const int nb = ceil_div(n, kBlock);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, heads, n, d) || !make_map(&mk, k, heads, n, d) ||
      !make_map(&mv, v, heads, n, d))
    return PISA_ERR_CUDA;
  const int smem = (d == 128 ? Smem<128>::MASK : Smem<64>::MASK) + 4 * ceil_div(nb, 32) * 4 + 1024;
  const dim3 grid(ceil_div(n, CTA_ROWS), heads);
  auto run = [&](auto kern) -> int {
    PISA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    kern<<<grid, NUM_THREADS, smem, stream>>>(mq, mk, mv, n, nb, scale, idx, cnt, max_sel, out,
                                              out_bf16, dev_status, spread);
    PISA_CHECK_LAUNCH();
    return PISA_OK;
  };
  if (d == 128)
    return spread ? run(forward_tc_kernel<128, true>) : run(forward_tc_kernel<128, false>);
  return spread ? run(forward_tc_kernel<64, true>) : run(forward_tc_kernel<64, false>);
}

}  // namespace pisa
