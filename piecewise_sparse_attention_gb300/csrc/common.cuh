// Shared device/host helpers of the PISA library (no kernels here).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pisa.h"

namespace pisa {

constexpr int kBlock = 64;  // tokens per block

// ---------------------------------------------------------------------------
// Run-time error reporting from device code: first error wins, no trap.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Loading 16-byte chunks of bf16 / float32 rows as float32.
// ---------------------------------------------------------------------------
template <typename T>
struct Chunk;

template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* f) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

template <>
struct Chunk<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void load(const float* p, float* f) {
    float4 u = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
};

// ---------------------------------------------------------------------------
// Error-free transformations (Knuth TwoSum, FMA-based TwoProduct) used for
// compensated sums and double-float dot products.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  // requires |a| >= |b| (or a == 0)
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// Compensated accumulator: value = s + c, with c collecting rounding errors.
struct CSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    float t, e;
    two_sum(s, x, t, e);
    s = t;
    c = __fadd_rn(c, e);
  }
  __device__ __forceinline__ void merge(const CSum& o) {
    float t, e;
    two_sum(s, o.s, t, e);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, o.c));
  }
  __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

// Double-float accumulator of a dot product (~2^-44 relative accuracy).
struct DFloat {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void fma_acc(float a, float b) {
    float p = __fmul_rn(a, b);
    float pe = __fmaf_rn(a, b, -p);  // exact product error
    float s, e;
    two_sum(hi, p, s, e);
    e = __fadd_rn(e, __fadd_rn(lo, pe));
    fast_two_sum(s, e, hi, lo);
  }
  __device__ __forceinline__ void merge(float ohi, float olo) {
    float s, e;
    two_sum(hi, ohi, s, e);
    e = __fadd_rn(e, __fadd_rn(lo, olo));
    fast_two_sum(s, e, hi, lo);
  }
};

// Order-preserving map float -> uint32 (larger float => larger integer);
// -0 is folded onto +0.
__device__ __forceinline__ uint32_t ord32(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// 64-bit key of a normalised double-float value (hi = fl(hi + lo)):
// lexicographic (hi, lo) order equals value order.
__device__ __forceinline__ uint64_t dfloat_key(float hi, float lo) {
  return (static_cast<uint64_t>(ord32(hi)) << 32) | ord32(lo);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace pisa

namespace pisa {
// Records a description of the last CUDA failure of the calling host thread
// (read back through pisa_last_error()); returns PISA_ERR_CUDA.
int cuda_fail(const char* what, int code, const char* detail);
// Records a printf-style description for pisa_last_error() (no status change).
void note_error(const char* fmt, ...);
}  // namespace pisa

// Launch-error check for host code: returns PISA_ERR_CUDA on failure.
#define PISA_CHECK_LAUNCH()                                                         \
  do {                                                                              \
    cudaError_t err__ = cudaGetLastError();                                         \
    if (err__ != cudaSuccess)                                                       \
      return ::pisa::cuda_fail(__func__, static_cast<int>(err__), cudaGetErrorString(err__)); \
  } while (0)

#define PISA_CUDA_TRY(call)                                                         \
  do {                                                                              \
    cudaError_t err__ = (call);                                                     \
    if (err__ != cudaSuccess)                                                       \
      return ::pisa::cuda_fail(#call, static_cast<int>(err__), cudaGetErrorString(err__)); \
  } while (0)
