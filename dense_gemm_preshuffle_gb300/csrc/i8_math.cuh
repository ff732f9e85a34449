// Exact integer arithmetic on the 16-bit tensor path, shared by the INT8
// weight-streaming kernels: int8 activations and offset-binary weight bytes
// become exact fp16 images, m16n8k16 MMAs accumulate one 128-element K tile
// exactly in fp32, and each tile's sums return to int32 with one FMA.
#pragma once
#include <cstdint>

namespace gp {

// Offset-binary bytes u -> fp16 subnormals u * 2^-24 (bit pattern 0x00uu):
// lo holds bytes 0 and 1, hi bytes 2 and 3.
__device__ __forceinline__ void u8x4_to_f16x2_sub(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0u));
}

// x = f * 2^24 is an integer with |x| < 2^22: x + 1.5 * 2^23 lies in
// [2^23, 2^24), where the fp32 ulp is 1, so the FMA is exact and the low
// bits of the result are x + 0x400000.
__device__ __forceinline__ int scaled_to_int(float f) {
  return (int)(__float_as_uint(__fmaf_rn(f, 16777216.0f, 12582912.0f)) - 0x4B400000u);
}

__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // each byte b -> b + 128 in [0, 255]
  uint32_t l, h;
  // fp16 0x64XX is exactly 1024 + XX
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(l) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(h) : "r"(u), "r"(0x64646464u));
  // subtract 1024 + 128 (fp16 0x6480): exact, the results are integers in [-128, 127]
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// Pure function of its register operands (no side effects), so ptxas may
// interleave independent accumulator chains freely.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace gp
