// Device-side MXFP8 helpers: E8M0 scale from a group amax, FP8 encoding, tiled scale offsets,
// bf16 packing.  Shared by the quantisers and the GEMM epilogues.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace moebwd {

// OCP MX rule: byte = clamp(floor(log2(amax)) - emax + 127, 0, 254) with floor(log2(amax)) read
// from the binary exponent field (a zero / subnormal amax gives byte 0); emax = 8 (e4m3), 15 (e5m2).
__device__ __forceinline__ uint32_t e8m0_byte(uint32_t amax_bits, int fmt) {
  const int e = (int)((amax_bits >> 23) & 0xFFu);
  const int b = e - (fmt == MOE_FP8_E4M3 ? 8 : 15);
  return (uint32_t)(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// 2^(127 - byte) as a float (byte <= 246 for finite inputs, so this is a normal number).
__device__ __forceinline__ float e8m0_inv_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

// Byte offset of the scale of element (r, c) of an [R, C] matrix quantised along C, in the tiled
// layout consumed by the block-scaled MMA: 512-byte atoms of 128 rows x 4 groups, atom grid
// row-major over (R/128, C/128), inside an atom (r%32)*16 + ((r%128)/32)*4 + (c/32)%4.
__device__ __forceinline__ int64_t sf_tiled_offset(int64_t r, int64_t c, int64_t C) {
  return ((r >> 7) * (C >> 7) + (c >> 7)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + ((c >> 5) & 3);
}

// max |v[i]| over N values (N a power of two) as a tree of pairwise maxima: log2(N) dependent steps
// instead of N (the maximum is exact in any order).
template <int N>
__device__ __forceinline__ float amax_tree(const float* v) {
  static_assert((N & (N - 1)) == 0, "power of two");
  if constexpr (N == 1) {
    return fabsf(v[0]);
  } else {
    return fmaxf(amax_tree<N / 2>(v), amax_tree<N / 2>(v + N / 2));
  }
}

// One 32-byte global store (a whole L2 sector); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_32b(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                              uint32_t w4, uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2),
               "r"(w3), "r"(w4), "r"(w5), "r"(w6), "r"(w7)
               : "memory");
}

// The same 32 bytes where p may be only 16-byte aligned (caller-owned outputs): two 16-byte stores then.
__device__ __forceinline__ void st_global_32b_or_halves(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                                        uint32_t w4, uint32_t w5, uint32_t w6, uint32_t w7) {
  if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
    st_global_32b(p, w0, w1, w2, w3, w4, w5, w6, w7);
  } else {
    reinterpret_cast<uint4*>(p)[0] = make_uint4(w0, w1, w2, w3);
    reinterpret_cast<uint4*>(p)[1] = make_uint4(w4, w5, w6, w7);
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)float_to_bf16_bits(lo) | ((uint32_t)float_to_bf16_bits(hi) << 16);
}

// Four FP8 codes (little-endian in one word) of a, b, c, d: two paired round-to-nearest-even
// saturating conversions (the sign is kept: a negative value rounding to zero gives -0, 0x80).
__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d, int fmt) {
  uint16_t lo, hi;
  if (fmt == MOE_FP8_E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  }
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// fp8x4 with the format fixed at compile time.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4_t(float a, float b, float c, float d) {
  uint16_t lo, hi;
  if constexpr (FMT == MOE_FP8_E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  }
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Two fp32 values in one 64-bit register for the paired fp32 arithmetic of sm_100-family SMs: each
// add / mul / fma of .f32x2 performs two round-to-nearest-even operations, each exactly the scalar
// one, in one instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_splat(float x) { return f2_pack(x, x); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Four FP8 codes of (a, b, c, d) * inv (inv a power of two: the products are exact), the products
// formed two at a time.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4_scaled(float a, float b, float c, float d, uint64_t inv2) {
  float x0, x1, x2, x3;
  f2_unpack(f2_mul(f2_pack(a, b), inv2), x0, x1);
  f2_unpack(f2_mul(f2_pack(c, d), inv2), x2, x3);
  return fp8x4_t<FMT>(x0, x1, x2, x3);
}

// Quantise 32 values of one group into 32 FP8 codes (packed little-endian into 8 words) and
// return the scale byte.
__device__ __forceinline__ uint32_t quantize_group32(const float (&v)[32], int fmt, uint32_t (&w)[8]) {
  const float am = amax_tree<32>(v);
  const uint32_t byte = e8m0_byte(__float_as_uint(am), fmt);
  const float inv = e8m0_inv_scale(byte);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j] = fp8x4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv, fmt);
  return byte;
}

// quantize_group32 with the format fixed at compile time.
template <int FMT>
__device__ __forceinline__ uint32_t quantize_group32_t(const float (&v)[32], uint32_t (&w)[8]) {
  const float am = amax_tree<32>(v);
  const uint32_t byte = e8m0_byte(__float_as_uint(am), FMT);
  const uint64_t inv2 = f2_splat(e8m0_inv_scale(byte));
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = fp8x4_scaled<FMT>(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3], inv2);
  return byte;
}

// quantize_group32_t with the group's amax given as the bits of an fp32 value (only its exponent
// field is used).
template <int FMT>
__device__ __forceinline__ uint32_t quantize_group32_am(const float (&v)[32], uint32_t am_bits, uint32_t (&w)[8]) {
  const uint32_t byte = e8m0_byte(am_bits, FMT);
  const uint64_t inv2 = f2_splat(e8m0_inv_scale(byte));
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = fp8x4_scaled<FMT>(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3], inv2);
  return byte;
}

// Per half, max |x| over 32 words of two bf16 values each (a tree of max.xorsign.abs.bf16x2: the
// magnitudes are maxima of magnitudes at every step, the sign bits are cleared at the end).  The
// maximum of bf16 magnitudes is itself a bf16 value, so this is the fp32 amax of either half exactly.
__device__ __forceinline__ uint32_t bf16x2_absmax32(const uint32_t (&w)[32]) {
  uint32_t t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(t[i]) : "r"(w[i]), "r"(w[i + 16]));
#pragma unroll
  for (int n = 8; n > 0; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(t[i]) : "r"(t[i]), "r"(t[i + n]));
  return t[0] & 0x7FFF7FFFu;
}

}  // namespace moebwd
