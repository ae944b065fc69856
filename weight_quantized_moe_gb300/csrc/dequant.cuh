// Exact weight-code conversions shared by the expert GEMMs: 8-bit and
// packed 4-bit codes to f16 / bf16 pairs, built by placing each code under
// a fixed exponent and subtracting the offset (no int-to-float conversion
// instructions).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mq {
namespace dq {

// 8-bit codes x4 -> two f16x2 words, exact.  xm = 0x80808080 turns an
// int8 code into u = q + 128 (the sign bit flipped), xm = 0 keeps a uint8
// code u; the half with bits 0x64uu is 1024 + u, and subtracting
// zz = 1024 + z (z = 128, or the row's zero point) leaves u - z.
__device__ __forceinline__ void int8x4_to_f16x4(uint32_t w, uint32_t xm, uint32_t zz,
                                                uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ xm;
  const uint32_t v0 = __byte_perm(u, 0x64u, 0x4140);  // [u0, 0x64, u1, 0x64]
  const uint32_t v1 = __byte_perm(u, 0x64u, 0x4342);  // [u2, 0x64, u3, 0x64]
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(v0), "r"(zz));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(v1), "r"(zz));
}

// 16 codes -> 8 words of f16 pairs.
__device__ __forceinline__ void convert16(const uint4& v, uint32_t xm, uint32_t zz, uint32_t* w) {
  int8x4_to_f16x4(v.x, xm, zz, w[0], w[1]);
  int8x4_to_f16x4(v.y, xm, zz, w[2], w[3]);
  int8x4_to_f16x4(v.z, xm, zz, w[4], w[5]);
  int8x4_to_f16x4(v.w, xm, zz, w[6], w[7]);
}

// (a0 - b, a1 - b) as one paired f32 subtraction (sm_100 family).
__device__ __forceinline__ void f32x2_sub(float a0, float a1, float b, float& r0, float& r1) {
  asm("{.reg .b64 xa, xb, xd;\n\t"
      "mov.b64 xa, {%2, %3};\n\t"
      "mov.b64 xb, {%4, %4};\n\t"
      "sub.rn.f32x2 xd, xa, xb;\n\t"
      "mov.b64 {%0, %1}, xd;}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b));
}

// 8-bit codes x4 -> two bf16x2 words, exact.  u = code ^ xm as above; the
// float with bits 0x4B0000uu is 2^23 + u, and subtracting zf = 2^23 + z
// leaves u - z exactly; |u - z| < 256 has at most 8 significant bits, so the
// top 16 bits of that float are the exact bfloat16.  (Measured faster than
// building 128 + (u & 127) and 128 or 256 as bfloat16 and subtracting those.)
__device__ __forceinline__ void int8x4_to_bf16x4(uint32_t w, uint32_t xm, float zf, uint32_t& lo,
                                                 uint32_t& hi) {
  const uint32_t u = w ^ xm;
  float f0, f1, f2, f3;
  f32x2_sub(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
            __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)), zf, f0, f1);
  f32x2_sub(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
            __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)), zf, f2, f3);
  lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
  hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

// 16 codes -> 8 words of bf16 pairs.
__device__ __forceinline__ void convert16_bf16(const uint4& v, uint32_t xm, float zf, uint32_t* w) {
  int8x4_to_bf16x4(v.x, xm, zf, w[0], w[1]);
  int8x4_to_bf16x4(v.y, xm, zf, w[2], w[3]);
  int8x4_to_bf16x4(v.z, xm, zf, w[4], w[5]);
  int8x4_to_bf16x4(v.w, xm, zf, w[6], w[7]);
}

// Position of K index i inside its octet under the order [0,4,1,5,2,6,3,7]
// (index c < 4 at 2c, index c + 4 at 2c + 1).
__host__ __device__ __forceinline__ int permute_octet(int i) {
  const int o = i & 7;
  return (i & ~7) | (o < 4 ? 2 * o : 2 * (o - 4) + 1);
}

// uint4 -> f16, one 32-bit word w = 8 codes k0..k7 of one K octet (two per
// byte, even index in the low nibble).  Word j of the result holds codes
// (k_j, k_{j+4}): one mask places both under the f16 exponent of 1024, so
// within every K octet the tensor-memory order is [0,4,1,5,2,6,3,7]; the
// activations are laid out in the same order, which leaves the dot product
// unchanged.  Each half becomes 1024 + q (exact); subtracting zz = 1024 + z
// gives q - z exactly; multiplying by the f16 group scale ss rounds once.
__device__ __forceinline__ void uint4x8_to_f16(uint32_t w, uint32_t zz, uint32_t ss, uint32_t* o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(zz));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(d), "r"(ss));
  }
}

// uint4 -> 16-bit pairs without a scale: word j of o holds codes
// (k_j, k_{j+4}) of the K octet in w, minus the zero point.  `magic` is the
// 16-bit pattern of the exponent that makes the low nibble the units digit
// (0x6400 = 1024 in f16, 0x4300 = 128 in bf16) broadcast to both halves;
// zz is (magic | z) in both halves.  The subtraction is exact (|q - z| <= 15).
template <bool BF16>
__device__ __forceinline__ void uint4x8_to_16(uint32_t w, uint32_t zz, uint32_t* o) {
  constexpr uint32_t magic = BF16 ? 0x43004300u : 0x64006400u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | magic;
    if constexpr (BF16) asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(v), "r"(zz));
    else asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(v), "r"(zz));
  }
}

}  // namespace dq
}  // namespace mq
