// Diagnostic kernel for the tensor-core building blocks (declared in
// include/pisa_selftest.h): 128x128x128 bf16 products computed four ways with
// tcgen05.mma -- B K-major from shared memory, B MN-major from shared memory,
// A read from tensor memory, and A MN-major (transposed) from shared memory --
// after TMA loads with 128-byte swizzle. A GPU test compares the three results with a reference product, so
// the descriptor encodings used by the attention kernel are checked in
// isolation. Mode 1 instead waits on an mbarrier that nothing signals and must
// come back with PISA_ERR_TIMEOUT in the status word (bounded-wait check).
#include "../../include/pisa_selftest.h"
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace pisa {
namespace {

constexpr int kPanel = 128 * 128;  // bytes of one [128 rows][64 bf16] panel
constexpr int kSmem = 6 * kPanel + 1024 + 256;

__global__ void __launch_bounds__(128, 1)
selftest_kernel(const __grid_constant__ CUtensorMap map_a,
                const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_bt, const __nv_bfloat16* a_glob,
                float* out, int mode, int32_t* status) {
  extern __shared__ unsigned char raw[];
  const uint32_t base_s = tc::smem_u32(raw);
  unsigned char* smem = raw + ((1024 - (base_s & 1023)) & 1023);
  unsigned char* sA = smem;
  unsigned char* sB = smem + 2 * kPanel;
  unsigned char* sBt = smem + 4 * kPanel;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * kPanel);
  uint64_t* tma_bar = bars;
  uint64_t* mma_bar = bars + 1;
  uint64_t* never_bar = bars + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid / 32;
  if (tid == 0) {
    abort_flag = 0;
    tc::mbar_init(tma_bar, 1);
    tc::mbar_init(mma_bar, 1);
    tc::mbar_init(never_bar, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 512);  // 4 accumulators of 128 columns
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (mode == 1) {
    if (tid == 0 && !tc::mbar_wait(never_bar, 0, &abort_flag, 1000000)) {
      abort_flag = 1;
      report(status, PISA_ERR_TIMEOUT);
    }
  } else {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(tma_bar, 6 * kPanel);
      for (int p = 0; p < 2; ++p) {
        tc::tma_load_2d(sA + p * kPanel, &map_a, 64 * p, 0, tma_bar);
        tc::tma_load_2d(sB + p * kPanel, &map_b, 64 * p, 0, tma_bar);
        tc::tma_load_2d(sBt + p * kPanel, &map_bt, 64 * p, 0, tma_bar);
      }
    }
    // A into TMEM columns [384, 448): row tid, bf16 pairs packed low-first
    {
      uint32_t r[32];
      const uint32_t* arow = reinterpret_cast<const uint32_t*>(a_glob + tid * 128);
      for (int half = 0; half < 2; ++half) {
        for (int c = 0; c < 32; ++c) r[c] = arow[half * 32 + c];
        tc::tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 384 + 32 * half, r);
      }
      tc::tmem_wait_st();
    }
    bool ok = tc::mbar_wait(tma_bar, 0, &abort_flag, 2000000000LL);
    if (!ok && tid == 0) {
      abort_flag = 1;
      report(status, PISA_ERR_TIMEOUT);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 0 && !abort_flag) {
      const uint32_t idesc_k = tc::idesc_bf16_f32(128, 128, false);
      const uint32_t idesc_mn = tc::idesc_bf16_f32(128, 128, true);
      const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB), bt0 = tc::smem_u32(sBt);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * kPanel + (ks % 4) * 32;
        const uint64_t ad = tc::smem_desc_sw128(a0 + off, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + off, 16, 1024);
        const uint64_t btd = tc::smem_desc_sw128(bt0 + ks * 2048, kPanel, 1024);
        tc::mma_ss(tmem + 0, ad, bd, idesc_k, ks > 0);
        tc::mma_ss(tmem + 128, ad, btd, idesc_mn, ks > 0);
        tc::mma_ts(tmem + 256, tmem + 384 + 8 * ks, btd, idesc_mn, ks > 0);
      }
      tc::mma_commit(mma_bar);
    }
    if (!abort_flag) {
      ok = tc::mbar_wait(mma_bar, 0, &abort_flag, 2000000000LL);
      if (!ok) {
        abort_flag = 1;
        report(status, PISA_ERR_TIMEOUT);
      }
    }
    tc::tc_fence_after();
    if (!abort_flag) {
      for (int which = 0; which < 3; ++which) {
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + which * 128 + 32 * c, r);
          tc::tmem_wait_ld();
          float* o = out + (static_cast<size_t>(which) * 128 + tid) * 128 + 32 * c;
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
        }
      }
    }
    // second phase: A read MN-major (a^T) from shared memory into columns
    // [0, 128) once the first results are out of tensor memory
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 0 && !abort_flag) {
      const uint32_t idesc_mnmn = tc::idesc_bf16_f32(128, 128, true) | (1u << 15);
      const uint32_t a0 = tc::smem_u32(sA), bt0 = tc::smem_u32(sBt);
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t atd = tc::smem_desc_sw128(a0 + ks * 2048, kPanel, 1024);
        const uint64_t btd = tc::smem_desc_sw128(bt0 + ks * 2048, kPanel, 1024);
        tc::mma_ss(tmem + 0, atd, btd, idesc_mnmn, ks > 0);
      }
      tc::mma_commit(mma_bar);
    }
    if (!abort_flag) {
      if (!tc::mbar_wait(mma_bar, 1, &abort_flag, 2000000000LL)) {
        abort_flag = 1;
        report(status, PISA_ERR_TIMEOUT);
      }
    }
    tc::tc_fence_after();
    if (__all_sync(0xffffffffu, !abort_flag)) {
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * c, r);
        tc::tmem_wait_ld();
        float* o = out + (static_cast<size_t>(3) * 128 + tid) * 128 + 32 * c;
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

bool make_2d(CUtensorMap* m, const void* p) {
  const uint64_t dims[2] = {128, 128};
  const uint64_t strides[1] = {256};
  const uint32_t box[2] = {64, 128};
  return make_tmap_bf16(m, p, 2, dims, strides, box);
}

}  // namespace
}  // namespace pisa

extern "C" int pisa_selftest_tc(const void* a, const void* b, const void* bt, float* out, int mode,
                                int32_t* dev_status, void* stream) {
  using namespace pisa;
  if (!a || !b || !bt || !out || (mode != 0 && mode != 1)) return PISA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
       reinterpret_cast<uintptr_t>(bt)) & 15u)
    return PISA_ERR_INVALID_ARG;
  CUtensorMap ma, mb, mbt;
  if (!make_2d(&ma, a) || !make_2d(&mb, b) || !make_2d(&mbt, bt)) return PISA_ERR_CUDA;
  PISA_CUDA_TRY(cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  selftest_kernel<<<1, 128, kSmem, static_cast<cudaStream_t>(stream)>>>(
      ma, mb, mbt, static_cast<const __nv_bfloat16*>(a), out, mode, dev_status);
  PISA_CHECK_LAUNCH();
  return PISA_OK;
}
