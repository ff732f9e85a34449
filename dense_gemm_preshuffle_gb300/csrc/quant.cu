// Activation quantisers in front of the GEMM: the operand recipes the
// workloads state ("GEMM Optimization Guide", section 8.2: per-token fp32
// scales for FP8; one UE8M0 byte per 32 K-elements for MXFP4), on the GPU.
//
//   - E4M3, per row: s = amax(|x|) / 448 (1 when the row is all zero), then
//     q = E4M3FN(x / s), round to nearest even, saturating at +-448.  Both
//     divisions are IEEE fp32 (this file is built without fast math, so
//     neither division nor denormal flushing can move a code).  One CTA per
//     row: a first pass reduces amax, a second pass writes the codes.  Rows
//     of up to 8192 elements stay in registers between the passes (32
//     values a thread); longer rows are read again, from L2.
//   - MXFP4, per 32-element block along K: e = the smallest integer with
//     amax <= 6 * 2^e.  With amax = f * 2^x (f in [0.5, 1)) that is x - 3
//     when f <= 0.75, else x - 2.  Then q = E2M1(x * 2^-e), round to
//     nearest even, saturating at +-6.  Two codes per byte, even k in the
//     low nibble; the exponent byte is e + 127.  Four lanes share a block
//     (8 elements each, two shuffles for the amax), so loads and stores are
//     fully coalesced.
//   - The E4M3 quotients come from a reciprocal multiply wherever that
//     provably gives the same code as the IEEE quotient (see
//     quotient_for_e4m3), else from the division itself.
// Both are HBM-bound: x is read once from DRAM, the codes written once.
#include <cuda_bf16.h>

#include "kernels.h"

namespace gp {

namespace {

template <typename XT>
__device__ __forceinline__ void load4(const XT* p, float (&v)[4]);

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
}

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(u.x << 16), v[1] = __uint_as_float(u.x & 0xFFFF0000u);
  v[2] = __uint_as_float(u.y << 16), v[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// One 16-byte load: 4 fp32 or 8 bf16 values (EV of them).
template <typename XT>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int EV = 4;
  __device__ __forceinline__ static void load(const float* p, float (&v)[4]) { load4<float>(p, v); }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int EV = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) v[2 * j] = __uint_as_float(w[j] << 16), v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
};

// Two fp32 values -> two E4M3 codes: lo in bits 0-7, hi in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values -> two E2M1 codes: lo in bits 0-3, hi in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// fp32(x / s) where only its E4M3 code matters.  y = x * (1/s) (both
// rounded to nearest) is within 2 fp32 ulps of x / s.  Two values that
// close round to the same E4M3 code unless an E4M3 rounding midpoint lies
// between them.  In a normal E4M3 binade the midpoints sit where the low 20
// fraction bits of an fp32 are 0x80000.  So y is used when those bits are
// more than 4 ulps from 0x80000 and |y| >= 2^-6 (E4M3's normal range; a
// power of two is itself an E4M3 value, so crossing one changes no code);
// the rest take the IEEE division itself.  The code is that of fp32(x / s)
// in every case.
__device__ __forceinline__ float quotient_for_e4m3(float x, float s, float inv) {
  const float y = x * inv;
  const uint32_t frac20 = __float_as_uint(y) & 0xFFFFFu;
  const uint32_t dist = frac20 > 0x80000u ? frac20 - 0x80000u : 0x80000u - frac20;
  // |x / s| <= 448 (1 + 2^-23); a larger y means 1/s overflowed (s below
  // 2^-128), so it too takes the division.
  if (dist > 4u && fabsf(y) >= 0.015625f && fabsf(y) <= 512.0f) return y;
  return __fdiv_rn(x, s);
}

__device__ __forceinline__ float block_amax(float amax, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  __syncthreads();  // red is reused by the next row
  return amax;
}

// Rows of up to 256 * VPT * EV elements: each thread keeps its VPT 16-byte
// vectors in registers between the amax pass and the quantising pass, so
// the row is read from memory once.
template <typename XT, int VPT>
__global__ void __launch_bounds__(256, 4) quant_e4m3_rows_reg_kernel(const XT* __restrict__ X, int64_t M, int64_t K,
                                                                  uint8_t* __restrict__ Q, float* __restrict__ S) {
  constexpr int EV = Vec16<XT>::EV;
  __shared__ float red[8];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const XT* x = X + row * K;
    float v[VPT][EV];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t i = ((int64_t)j * blockDim.x + threadIdx.x) * EV;
      if (i < K) {
        Vec16<XT>::load(x + i, v[j]);
#pragma unroll
        for (int e = 0; e < EV; ++e) amax = fmaxf(amax, fabsf(v[j][e]));
      }
    }
    amax = block_amax(amax, red);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const float inv = __frcp_rn(s);
    if (threadIdx.x == 0) S[row] = s;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t i = ((int64_t)j * blockDim.x + threadIdx.x) * EV;
      if (i < K) {
        uint32_t w[EV / 4];
#pragma unroll
        for (int k = 0; k < EV / 4; ++k)
          w[k] = e4m3x2(quotient_for_e4m3(v[j][4 * k], s, inv), quotient_for_e4m3(v[j][4 * k + 1], s, inv)) |
                 (e4m3x2(quotient_for_e4m3(v[j][4 * k + 2], s, inv), quotient_for_e4m3(v[j][4 * k + 3], s, inv))
                  << 16);
        if constexpr (EV == 4)
          *reinterpret_cast<uint32_t*>(Q + row * K + i) = w[0];
        else
          *reinterpret_cast<uint2*>(Q + row * K + i) = make_uint2(w[0], w[1]);
      }
    }
  }
}

// Longer rows: the quantising pass reads the row again (from L2).
template <typename XT>
__global__ void __launch_bounds__(256) quant_e4m3_rows_kernel(const XT* __restrict__ X, int64_t M, int64_t K,
                                                              uint8_t* __restrict__ Q, float* __restrict__ S) {
  __shared__ float red[8];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const XT* x = X + row * K;
    float amax = 0.0f;
    for (int64_t i = threadIdx.x * 4; i < K; i += 4 * blockDim.x) {
      float v[4];
      load4<XT>(x + i, v);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    amax = block_amax(amax, red);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) S[row] = s;
    for (int64_t i = threadIdx.x * 4; i < K; i += 4 * blockDim.x) {
      float v[4];
      load4<XT>(x + i, v);
      const uint32_t lo = e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s));
      const uint32_t hi = e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
      *reinterpret_cast<uint32_t*>(Q + row * K + i) = lo | (hi << 16);
    }
  }
}

// grid.x covers the 8-element groups of a row (256 per CTA); grid.y strides
// over groups of MX_ROWS rows, whose loads a thread issues together (more
// bytes in flight).  All index arithmetic is division-free.
constexpr int MX_ROWS = 4;

template <typename XT>
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const XT* __restrict__ X, int64_t M, int K,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ E) {
  const int per_row = K / 8;  // 8-element groups per row; 4 groups per 32-element block
  const int c8 = blockIdx.x * blockDim.x + threadIdx.x;
  // A 4-lane group is entirely inside or outside the row (per_row % 4 == 0),
  // and every lane takes part in the shuffles.
  const bool active = c8 < per_row;
  for (int64_t row0 = (int64_t)blockIdx.y * MX_ROWS; row0 < M; row0 += (int64_t)gridDim.y * MX_ROWS) {
    float v[MX_ROWS][8];
#pragma unroll
    for (int r = 0; r < MX_ROWS; ++r) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[r][j] = 0.0f;
      const int64_t row = row0 + r;
      if (active && row < M) {
        const XT* x = X + row * (int64_t)K + (int64_t)c8 * 8;
        if constexpr (Vec16<XT>::EV == 8) {
          Vec16<XT>::load(x, v[r]);
        } else {
          float a[4], b[4];
          load4<XT>(x, a);
          load4<XT>(x + 4, b);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[r][j] = a[j], v[r][4 + j] = b[j];
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MX_ROWS; ++r) {
      const int64_t row = row0 + r;
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[r][j]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int e = 0;
      if (amax > 0.0f) {
        int ex;
        const float f = frexpf(amax, &ex);  // amax = f * 2^ex exactly
        e = f <= 0.75f ? ex - 3 : ex - 2;
        e = e < -127 ? -127 : (e > 127 ? 127 : e);
      }
      // 2^-e: e lies in [-127, 126] for finite fp32 amax, so 2^-e is a normal float
      const float scale = __int_as_float((uint32_t)(127 - e) << 23);
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) packed |= e2m1x2(v[r][2 * j] * scale, v[r][2 * j + 1] * scale) << (8 * j);
      if (active && row < M) {
        *reinterpret_cast<uint32_t*>(Q + row * (int64_t)(K / 2) + (int64_t)c8 * 4) = packed;
        if ((c8 & 3) == 0) E[row * (int64_t)(K / 32) + c8 / 4] = (uint8_t)(e + 127);
      }
    }
  }
}

int grid_rows(int64_t M) { return (int)(M < 65535 * 4 ? M : 65535 * 4); }

}  // namespace

int quant_launch(const void* X, bool x_bf16, int64_t M, int64_t K, bool to_e2m1, void* Q, void* S,
                 cudaStream_t stream) {
  if (!to_e2m1) {
    const int grid = grid_rows(M);
    if (x_bf16 && K <= 256 * 4 * 8) {
      quant_e4m3_rows_reg_kernel<__nv_bfloat16, 4><<<grid, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(X), M, K, static_cast<uint8_t*>(Q), static_cast<float*>(S));
    } else if (!x_bf16 && K <= 256 * 8 * 4) {
      quant_e4m3_rows_reg_kernel<float, 8><<<grid, 256, 0, stream>>>(static_cast<const float*>(X), M, K,
                                                                      static_cast<uint8_t*>(Q),
                                                                      static_cast<float*>(S));
    } else if (x_bf16)
      quant_e4m3_rows_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), M, K,
                                                                       static_cast<uint8_t*>(Q),
                                                                       static_cast<float*>(S));
    else
      quant_e4m3_rows_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(X), M, K,
                                                               static_cast<uint8_t*>(Q), static_cast<float*>(S));
  } else {
    const int64_t groups = (M + MX_ROWS - 1) / MX_ROWS;
    const dim3 grid((unsigned)((K / 8 + 255) / 256), (unsigned)(groups < 65535 ? groups : 65535));
    if (x_bf16)
      quant_mxfp4_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), M, (int)K,
                                                                   static_cast<uint8_t*>(Q), static_cast<uint8_t*>(S));
    else
      quant_mxfp4_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(X), M, (int)K,
                                                           static_cast<uint8_t*>(Q), static_cast<uint8_t*>(S));
  }
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

}  // namespace gp
