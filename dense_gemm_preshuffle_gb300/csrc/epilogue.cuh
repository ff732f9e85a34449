// Fused epilogues of the float-output GEMMs ("Kernel Tuning Guide", section
// 6, Epilogue Strategies: "none", "bias", "bias_relu", "bias_silu",
// "bias_gelu").  For one row of 32 consecutive output columns:
//   v = acc * scale_a[m] * scale_b[n]   (scales when given)
//   v = v + bias[n]                     (fp32, one value per column)
//   v = act(v)                          ReLU max(v, 0); SiLU v / (1 + e^-v);
//                                       GELU 0.5 v (1 + erf(v / sqrt 2)),
//                                       erf by a published rational
//                                       approximation (|error| <= 1.5e-7)
// then rounded to bf16 or fp16 (RNE) in pairs.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace gp {

enum EpiAct : int { EPI_ACT_NONE = 0, EPI_ACT_RELU = 1, EPI_ACT_SILU = 2, EPI_ACT_GELU = 3 };

// GELU(x) = 0.5 x (1 + erf(x / sqrt 2)) through q = erfc(|x| / sqrt 2),
// evaluated with Abramowitz and Stegun, Handbook of Mathematical Functions,
// formula 7.1.26: erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^-z^2
// with t = 1 / (1 + p z), |error| <= 1.5e-7 for z >= 0.  Then
// GELU(x) = x - 0.5 x q for x >= 0 and 0.5 x q for x < 0, which keeps full
// relative accuracy in the negative tail (no cancellation).
__device__ __forceinline__ float epi_gelu(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  float poly = fmaf(t, 1.061405429f, -1.453152027f);
  poly = fmaf(t, poly, 1.421413741f);
  poly = fmaf(t, poly, -0.284496736f);
  poly = fmaf(t, poly, 0.254829592f);
  const float q = t * poly * __expf(-z * z);
  const float half_xq = 0.5f * x * q;
  return x >= 0.0f ? x - half_xq : half_xq;
}

__device__ __forceinline__ float epi_act(float x, int act) {
  switch (act) {
    case EPI_ACT_RELU: return fmaxf(x, 0.0f);
    case EPI_ACT_SILU: return __fdividef(x, 1.0f + __expf(-x));  // x -> -inf gives -0, x -> +inf gives x
    case EPI_ACT_GELU: return epi_gelu(x);
    default: return x;
  }
}

// v: the row's 32 fp32 values; sb, bias: the same 32 columns (16-byte
// aligned) or null; sa: the row scale (1 when absent); out_f16: round to
// IEEE binary16 instead of bf16 (both RNE).  BIAS_SMEM: bias points into
// shared memory (else global, read through the read-only path).
template <bool BIAS_SMEM = false>
__device__ __forceinline__ void epi_row32(float (&v)[32], float sa, const float* sb, const float* bias, int act,
                                          bool out_f16, uint32_t (&pk)[16]) {
  if (sb != nullptr) {
    const float4* sb4 = reinterpret_cast<const float4*>(sb);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 s4 = __ldg(sb4 + q);
      v[4 * q] = v[4 * q] * sa * s4.x;
      v[4 * q + 1] = v[4 * q + 1] * sa * s4.y;
      v[4 * q + 2] = v[4 * q + 2] * sa * s4.z;
      v[4 * q + 3] = v[4 * q + 3] * sa * s4.w;
    }
  }
  if (bias != nullptr) {
    const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 b = BIAS_SMEM ? b4[q] : __ldg(b4 + q);
      v[4 * q] += b.x;
      v[4 * q + 1] += b.y;
      v[4 * q + 2] += b.z;
      v[4 * q + 3] += b.w;
    }
    if (act != EPI_ACT_NONE) {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = epi_act(v[e], act);
    }
  }
  if (out_f16) {
#pragma unroll
    for (int q = 0; q < 16; ++q) pk[q] = pack_f16x2(v[2 * q], v[2 * q + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
  }
}

}  // namespace gp
