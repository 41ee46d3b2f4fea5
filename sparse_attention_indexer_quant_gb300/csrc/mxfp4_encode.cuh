// MXFP4 encoding of one 128-element vector by 16 threads (lanes
// [16g, 16g + 16) of a warp, 8 consecutive elements each), shared by the
// insert, q-quant, rotary q-quant and K-pool kernels.
//
// A block of 32 elements is four consecutive lanes: their max |x| is reduced
// with two butterfly shuffles on the integer bit patterns (for non-negative
// floats the bit order is the value order) and gives the block's UE8M0 byte.
// x * 2^-e is exact for every magnitude that can round to a nonzero code; the
// hardware convert rounds to nearest with ties to the even code, saturates at
// 6 and keeps the sign of a value that rounds to zero (the rule checked bit
// for bit against the oracle over every finite bf16 pattern); element 2i goes
// to the low nibble of byte i.
#pragma once

#include "common.cuh"

namespace idx {

// Encodes the 8 fp32 values x[0..7] held by this thread.  Returns the 4
// packed value bytes; *scales_word gets the vector's 4 scale bytes (valid in
// every lane of the 16-lane group).  All 32 lanes of the warp must call it.
__device__ __forceinline__ uint32_t encode8_f32(const float (&x)[8], uint32_t* scales_word) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(x[i]) & 0x7FFFFFFFu);
  // four consecutive lanes hold one block of 32
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  const uint32_t s = ue8m0_of_amax(amax);
  const float inv = inv_scale_of(s);
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = x[i] * inv;
  uint32_t packed;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(packed)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  // gather the 4 block scales of this vector: blocks live in lanes 0,4,8,12 of
  // the 16-lane group
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t base = lane & 16u;
  const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, s, base + 0);
  const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, s, base + 4);
  const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, s, base + 8);
  const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, s, base + 12);
  *scales_word = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
  return packed;
}

// The 8 bf16 values of this thread (as 4 x bf16x2 words, element 2i in the
// low half of word i) as fp32, exactly.
__device__ __forceinline__ void bf16x8_to_f32(uint4 raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// encode8_f32 of 8 bf16 values.
__device__ __forceinline__ uint32_t encode8(uint4 raw, uint32_t* scales_word) {
  float x[8];
  bf16x8_to_f32(raw, x);
  return encode8_f32(x, scales_word);
}

}  // namespace idx
