// Per-row register arithmetic shared by the tensor-core forward kernels: the
// softmax warps hold one query row's 128 scores (read from TMEM) in four
// 32-register chunks and work on them with these helpers.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace pisa {

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed float32 pairs (Blackwell f32x2 arithmetic: two lanes of work per
// instruction) held in a 64-bit register.
__device__ __forceinline__ uint64_t f2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2f(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Registers written by tcgen05.ld are only valid after tcgen05.wait::ld; this
// empty asm ties each of them to a point after the wait so no use is
// scheduled earlier.
__device__ __forceinline__ void after_wait(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// max / sum over the 64 fp32 values of one key block held in two 32-register
// chunks, with independent accumulators to shorten dependency chains
__device__ __forceinline__ float row_max64(const uint32_t (&x)[32], const uint32_t (&y)[32]) {
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmaxf(__uint_as_float(x[i]), __uint_as_float(y[i]));
#pragma unroll
  for (int i = 4; i < 32; ++i)
    m[i & 3] = max3(m[i & 3], __uint_as_float(x[i]), __uint_as_float(y[i]));
  return max3(m[0], m[1], fmaxf(m[2], m[3]));
}

__device__ __forceinline__ float row_sum64(const uint32_t (&x)[32], const uint32_t (&y)[32]) {
  uint64_t s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = add2(f2(x[2 * i], x[2 * i + 1]), f2(y[2 * i], y[2 * i + 1]));
#pragma unroll
  for (int i = 4; i < 16; ++i)
    s[i & 3] = add2(s[i & 3], add2(f2(x[2 * i], x[2 * i + 1]), f2(y[2 * i], y[2 * i + 1])));
  const uint64_t t = add2(add2(s[0], s[1]), add2(s[2], s[3]));
  float lo, hi;
  unf2(t, lo, hi);
  return lo + hi;
}

// keys nv..63 of a partial last block: -inf, so they neither raise the max
// nor add to the exact mass
__device__ __forceinline__ void mask_tail(uint32_t (&x)[32], uint32_t (&y)[32], int nv) {
  const uint32_t ninf = 0xff800000u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i >= nv) x[i] = ninf;
    if (32 + i >= nv) y[i] = ninf;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// The two bf16 values of a packed pair, widened exactly to a float32 pair.
// Weights that enter P V rounded to bf16 enter the softmax denominator in
// this rounded form too, so the output stays a weighted average of the
// values with the very weights the tensor cores used: a row dominated by one
// key (weight up to 2^20 under the lazy shift, where its bf16 rounding can
// reach 2^-9 of it) then returns that key's value without the rounding.
__device__ __forceinline__ uint64_t unpack_bf16x2(uint32_t pk) {
  return f2(pk << 16, pk & 0xffff0000u);
}

}  // namespace pisa
