// Activation quantisers in front of the GEMM: the operand recipes the
// workloads state ("GEMM Optimization Guide", section 8.2: per-token fp32
// scales for FP8; one UE8M0 byte per 32 K-elements for MXFP4), on the GPU.
//
//   - E4M3, per row: s = amax(|x|) / 448 (1 when the row is all zero), then
//     q = E4M3FN(x / s), round to nearest even, saturating at +-448.  Both
//     divisions are IEEE fp32 (this file is built without fast math, so
//     neither division nor denormal flushing can move a code).  One CTA
//     takes a row at a time: a first pass reduces amax, a second pass writes
//     the codes.  Between the passes the row stays on the SM: fp32 rows of
//     2-48 KiB in a shared-memory ring filled by bulk copies, shorter fp32
//     rows and bf16 rows of up to 8192 elements in registers.  Longer rows
//     are read again, from L2.
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
#include "ptx.cuh"

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

// One 16-byte vector: 4 fp32 or 8 bf16 values (EV of them), kept raw in
// registers and widened to fp32 (exactly) where used.
template <typename XT>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int EV = 4;
  __device__ __forceinline__ static void decode(const uint4& u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x), v[1] = __uint_as_float(u.y), v[2] = __uint_as_float(u.z), v[3] = __uint_as_float(u.w);
  }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int EV = 8;
  __device__ __forceinline__ static void decode(const uint4& u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) v[2 * j] = __uint_as_float(w[j] << 16), v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
};

__device__ __forceinline__ uint4 ld_vec16(const void* p) { return *reinterpret_cast<const uint4*>(p); }

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
//
// The test on y's bits: the low 20 fraction bits within 4 of 0x80000, or
// |y| outside [2^-6, 512] (bits 0x3C800000 .. 0x44000000; zero, NaN and
// the values past 512 fall outside).  |x / s| <= 448 (1 + 2^-23), so a y
// above 512 means 1/s overflowed (s below 2^-128).
__device__ __forceinline__ bool e4m3_needs_division(float y) {
  const uint32_t b = __float_as_uint(y);
  return ((b & 0xFFFFFu) - 0x7FFFCu) <= 8u || ((b & 0x7FFFFFFFu) - 0x3C800000u) > 0x07800000u;
}

__device__ __forceinline__ float quotient_for_e4m3(float x, float s, float inv) {
  const float y = x * inv;
  return e4m3_needs_division(y) ? __fdiv_rn(x, s) : y;
}

// The same test as e4m3_needs_division, negated and written with float
// compares.  The two agree on every fp32 bit pattern.  Inside the rarely
// taken branch of e4m3x4_div this spelling made the fp32 kernels faster
// (E4M3 8192 x 8192: 51.9 against 53.9 us); the bit test is faster where
// it runs on every value.
__device__ __forceinline__ bool e4m3_product_usable(float y) {
  const uint32_t frac20 = __float_as_uint(y) & 0xFFFFFu;
  const uint32_t dist = frac20 > 0x80000u ? frac20 - 0x80000u : 0x80000u - frac20;
  return dist > 4u && fabsf(y) >= 0.015625f && fabsf(y) <= 512.0f;
}

// The E4M3 codes of x[0..3] / s, packed little-endian into a word.  The
// per-value test of quotient_for_e4m3 is folded into one branch for the
// four values; a value that needs the division gets it, the others keep
// their product, so each code is still that of fp32(x / s).  Used by the
// fp32 kernels; the bf16 kernel was faster with the per-value form (44.0
// against 48.6 us).
__device__ __forceinline__ uint32_t e4m3x4_div(const float* x, float s, float inv) {
  float y[4];
  bool slow = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[i] = x[i] * inv;
    slow |= e4m3_needs_division(y[i]);
  }
  if (slow) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!e4m3_product_usable(y[i])) y[i] = __fdiv_rn(x[i], s);
  }
  return e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
}

// Programmatic dependent launch: the kernel waits for the previous kernel
// on the stream (which may write X, or read Q and S) before touching
// memory.  A persistent grid then lets the next kernel launch at once.
// Grids of many waves leave that to their exit, so that the next kernel's
// CTAs do not take SM slots from their own later waves (triggering early
// there took bf16 E4M3 8192 x 8192 from 46.2 to 49.5 us).  Back to back,
// MXFP4 from bf16 went from 16.9 to 16.4 us; the longer calls did not move.
template <bool PERSISTENT>
__device__ __forceinline__ void quant_prologue() {
  pdl_wait();
  if (PERSISTENT) pdl_launch_dependents();
}

// Max over the NW warps of a CTA of each of R values (red: R x NW floats).
template <int R, int NW>
__device__ __forceinline__ void block_amax(float (&amax)[R], float* red) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], o));
    if ((threadIdx.x & 31) == 0) red[r * NW + (threadIdx.x >> 5)] = amax[r];
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float m = red[r * NW];
#pragma unroll
    for (int w = 1; w < NW; ++w) m = fmaxf(m, red[r * NW + w]);
    amax[r] = m;
  }
  __syncthreads();  // red is reused by the next rows
}

// fp32 rows of up to 256 * 8 * 4 elements: each thread keeps its 8 float4
// vectors in registers between the amax pass and the quantising pass, so
// the row is read from memory once.  One CTA per row, four per SM.
__global__ void __launch_bounds__(256, 4) quant_e4m3_rows_f32_kernel(const float* __restrict__ X, int64_t M,
                                                                  int64_t K, uint8_t* __restrict__ Q,
                                                                  float* __restrict__ S) {
  quant_prologue<false>();
  constexpr int VPT = 8;
  __shared__ float red[8];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const float* x = X + row * K;
    float v[VPT][4];
    float amax[1] = {0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t i = ((int64_t)j * blockDim.x + threadIdx.x) * 4;
      if (i < K) {
        load4<float>(x + i, v[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) amax[0] = fmaxf(amax[0], fabsf(v[j][e]));
      }
    }
    block_amax<1, 8>(amax, red);
    const float s = amax[0] > 0.0f ? __fdiv_rn(amax[0], 448.0f) : 1.0f;
    const float inv = __frcp_rn(s);
    if (threadIdx.x == 0) S[row] = s;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t i = ((int64_t)j * blockDim.x + threadIdx.x) * 4;
      if (i < K)
        *reinterpret_cast<uint32_t*>(Q + row * K + i) = e4m3x4_div(v[j], s, inv);
    }
  }
}

// bf16 rows of up to THREADS * VPT * 8 elements, kept as raw 16-byte
// vectors (half the registers of fp32 values) and widened where used.  The
// bytes in flight per SM are the resident CTAs' rows, so the fewer
// registers buy more CTAs per SM (MINB).  Two rows a CTA at four CTAs per
// SM were slower than one row at six (bf16 8192 x 8192: 55 vs 46 us).
template <int THREADS, int VPT, int MINB>
__global__ void __launch_bounds__(THREADS, MINB) quant_e4m3_rows_bf16_kernel(const __nv_bfloat16* __restrict__ X,
                                                                          int64_t M, int64_t K,
                                                                          uint8_t* __restrict__ Q,
                                                                          float* __restrict__ S) {
  quant_prologue<false>();
  using V = Vec16<__nv_bfloat16>;
  constexpr int EV = V::EV;
  constexpr int NW = THREADS / 32;
  __shared__ float red[NW];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const __nv_bfloat16* x = X + row * K;
    uint4 raw[VPT];
    float amax[1] = {0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int i = (j * THREADS + (int)threadIdx.x) * EV;  // K <= THREADS * VPT * EV here
      if (i < K) raw[j] = ld_vec16(x + i);
    }
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int i = (j * THREADS + (int)threadIdx.x) * EV;
      if (i < K) {
        float v[EV];
        V::decode(raw[j], v);
#pragma unroll
        for (int e = 0; e < EV; ++e) amax[0] = fmaxf(amax[0], fabsf(v[e]));
      }
    }
    block_amax<1, NW>(amax, red);
    const float s = amax[0] > 0.0f ? __fdiv_rn(amax[0], 448.0f) : 1.0f;
    const float inv = __frcp_rn(s);
    if (threadIdx.x == 0) S[row] = s;
    uint8_t* q = Q + row * K;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int i = (j * THREADS + (int)threadIdx.x) * EV;
      if (i < K) {
        float v[EV];
        V::decode(raw[j], v);
        uint32_t w[2];
#pragma unroll
        for (int k = 0; k < 2; ++k)
          w[k] = e4m3x2(quotient_for_e4m3(v[4 * k], s, inv), quotient_for_e4m3(v[4 * k + 1], s, inv)) |
                 (e4m3x2(quotient_for_e4m3(v[4 * k + 2], s, inv), quotient_for_e4m3(v[4 * k + 3], s, inv)) << 16);
        *reinterpret_cast<uint2*>(q + i) = make_uint2(w[0], w[1]);
      }
    }
  }
}

// fp32 rows of 2-48 KiB staged through shared memory.  One bulk copy
// brings a whole row into a ring of NBUF row buffers.  While a CTA reduces
// and encodes one row, the copies of its next rows are in flight, so every
// resident CTA keeps reads outstanding through its compute phase and no
// registers hold the row.  A persistent grid (a whole number of CTAs per
// SM) walks the rows.  The arithmetic is that of the kernels above.
// Measured at 8192 x 8192: fp32 61.9 -> 55.0 us against the register
// kernel.  bf16 rows were slower staged (53-58 us with two or three
// buffers, against 49.6), so they keep the register kernel.
//
// Every wait is bounded.  After a timeout the CTA leaves as a whole (a
// barrier vote), once the copies still in flight have landed or their own
// bounded waits have run out.
template <typename XT, int NBUF>
__global__ void __launch_bounds__(256) quant_e4m3_rows_staged_kernel(const XT* __restrict__ X, int64_t M, int64_t K,
                                                                     uint8_t* __restrict__ Q, float* __restrict__ S,
                                                                     uint32_t* status, uint64_t limit_ns) {
  quant_prologue<true>();
  using V = Vec16<XT>;
  constexpr int EV = V::EV;
  constexpr int THREADS = 256, NW = THREADS / 32;
  extern __shared__ __align__(128) uint8_t rows[];
  __shared__ float red[NW];
  __shared__ uint64_t full[NBUF];
  __shared__ volatile int abort_flag;
  const uint32_t row_bytes = (uint32_t)(K * (int64_t)sizeof(XT));  // a multiple of 64 (K % 32 == 0)
  const int nvec = (int)(row_bytes / 16);
  if (threadIdx.x == 0) {
    for (int b = 0; b < NBUF; ++b) mbar_init(&full[b], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int b, int64_t row) {
    mbar_arrive_expect_tx(&full[b], row_bytes);
    bulk_load(rows + (size_t)b * row_bytes, X + row * K, row_bytes, &full[b]);
  };
  if (threadIdx.x == 0)
    for (int b = 0; b < NBUF; ++b) {
      const int64_t row = blockIdx.x + (int64_t)b * gridDim.x;
      if (row < M) issue(b, row);
    }
  int it = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, ++it) {
    const int b = it % NBUF;
    const bool ok = wait_bounded(&full[b], (uint32_t)(it / NBUF) & 1, &abort_flag, status, ST_TIMEOUT_CONSUMER,
                                 limit_ns);
    if (__syncthreads_or(!ok)) break;
    const uint4* buf = reinterpret_cast<const uint4*>(rows + (size_t)b * row_bytes);
    float amax[1] = {0.0f};
    for (int v = threadIdx.x; v < nvec; v += THREADS) {
      float x[EV];
      V::decode(buf[v], x);
#pragma unroll
      for (int e = 0; e < EV; ++e) amax[0] = fmaxf(amax[0], fabsf(x[e]));
    }
    block_amax<1, NW>(amax, red);
    const float s = amax[0] > 0.0f ? __fdiv_rn(amax[0], 448.0f) : 1.0f;
    const float inv = __frcp_rn(s);
    if (threadIdx.x == 0) S[row] = s;
    uint8_t* q = Q + row * K;
    for (int v = threadIdx.x; v < nvec; v += THREADS) {
      float x[EV];
      V::decode(buf[v], x);
      uint32_t w[EV / 4];
#pragma unroll
      for (int k = 0; k < EV / 4; ++k) w[k] = e4m3x4_div(x + 4 * k, s, inv);
      if constexpr (EV == 8)
        *reinterpret_cast<uint2*>(q + (size_t)v * 8) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t*>(q + (size_t)v * 4) = w[0];
    }
    __syncthreads();  // every thread is done with buffer b: refill it
    if (threadIdx.x == 0) {
      const int64_t next = row + (int64_t)NBUF * gridDim.x;
      if (next < M) issue(b, next);
    }
  }
  if (threadIdx.x == 0 && abort_flag) {
    // The copies of iterations it .. it + NBUF - 1 may still be in flight.
    volatile int never = 0;
    for (int j = 0; j < NBUF; ++j) {
      if ((int64_t)blockIdx.x + (int64_t)(it + j) * gridDim.x >= M) break;
      wait_bounded(&full[(it + j) % NBUF], (uint32_t)((it + j) / NBUF) & 1, &never, status, ST_TIMEOUT_DRAIN,
                   limit_ns);
    }
  }
}

constexpr int QS_NBUF = 2;
constexpr uint32_t QS_MIN_ROW = 2048, QS_MAX_ROW = 48 * 1024;  // fp32 row bytes that take the staged kernel

// Longer rows: the quantising pass reads the row again (from L2).
template <typename XT>
__global__ void __launch_bounds__(256) quant_e4m3_rows_kernel(const XT* __restrict__ X, int64_t M, int64_t K,
                                                              uint8_t* __restrict__ Q, float* __restrict__ S) {
  quant_prologue<false>();
  __shared__ float red[8];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const XT* x = X + row * K;
    float amax = 0.0f;
    for (int64_t i = threadIdx.x * 4; i < K; i += 4 * blockDim.x) {
      float v[4];
      load4<XT>(x + i, v);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    float am[1] = {amax};
    block_amax<1, 8>(am, red);
    amax = am[0];
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
// over groups of ROWS rows, whose loads a thread issues together (more
// bytes in flight).  All index arithmetic is division-free.
template <typename XT>
struct MxRows {
  static constexpr int value = 4;  // 8 rows of bf16 halve the grid and were slower (measured)
};

template <typename XT>
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const XT* __restrict__ X, int64_t M, int K,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ E) {
  quant_prologue<false>();
  constexpr int MX_ROWS = MxRows<XT>::value;
  constexpr int NV = 8 / Vec16<XT>::EV;  // 16-byte vectors per 8-element group
  const int per_row = K / 8;  // 8-element groups per row; 4 groups per 32-element block
  const int c8 = blockIdx.x * blockDim.x + threadIdx.x;
  // A 4-lane group is entirely inside or outside the row (per_row % 4 == 0),
  // and every lane takes part in the shuffles.
  const bool active = c8 < per_row;
  for (int64_t row0 = (int64_t)blockIdx.y * MX_ROWS; row0 < M; row0 += (int64_t)gridDim.y * MX_ROWS) {
    uint4 raw[MX_ROWS][NV];
#pragma unroll
    for (int r = 0; r < MX_ROWS; ++r) {
      const int64_t row = row0 + r;
#pragma unroll
      for (int q = 0; q < NV; ++q) raw[r][q] = make_uint4(0u, 0u, 0u, 0u);
      if (active && row < M) {
        const XT* x = X + row * (int64_t)K + (int64_t)c8 * 8;
#pragma unroll
        for (int q = 0; q < NV; ++q) raw[r][q] = ld_vec16(x + q * Vec16<XT>::EV);
      }
    }
#pragma unroll
    for (int r = 0; r < MX_ROWS; ++r) {
      const int64_t row = row0 + r;
      float v[8];
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        float t[Vec16<XT>::EV];
        Vec16<XT>::decode(raw[r][q], t);
#pragma unroll
        for (int e = 0; e < Vec16<XT>::EV; ++e) v[q * Vec16<XT>::EV + e] = t[e];
      }
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
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
      for (int j = 0; j < 4; ++j) packed |= e2m1x2(v[2 * j] * scale, v[2 * j + 1] * scale) << (8 * j);
      if (active && row < M) {
        *reinterpret_cast<uint32_t*>(Q + row * (int64_t)(K / 2) + (int64_t)c8 * 4) = packed;
        if ((c8 & 3) == 0) E[row * (int64_t)(K / 32) + c8 / 4] = (uint8_t)(e + 127);
      }
    }
  }
}

// bf16 rows of up to 8192: 256 threads x 4 vectors, six CTAs per SM (the
// best of 256 x 4 at 5-7 CTAs and 128 x 8 at 8-12, measured at 8192 x 8192)
constexpr int QB_THREADS = 256, QB_VPT = 4, QB_MINB = 6;

int grid_rows(int64_t M) { return (int)(M < 65535 * 4 ? M : 65535 * 4); }

// Every quantiser launch carries the programmatic-stream-serialisation
// attribute (see quant_prologue).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

// The staged kernel over a persistent grid: as many CTAs per SM as shared
// memory (228 KiB an SM, 1 KiB reserved per CTA) and threads allow.
template <typename XT>
int launch_staged(const XT* X, int64_t M, int64_t K, uint8_t* Q, float* S, int num_sms, uint32_t* status,
                  uint64_t limit_ns, cudaStream_t stream) {
  constexpr int NBUF = QS_NBUF;
  auto kern = quant_e4m3_rows_staged_kernel<XT, NBUF>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, (int)(NBUF * QS_MAX_ROW), 100); rc != GP_OK) return rc;
  const size_t smem = (size_t)NBUF * (size_t)K * sizeof(XT);
  int per_sm = (int)((228 * 1024) / (smem + 1024 + 256));
  per_sm = per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm);
  const int64_t ctas = (int64_t)num_sms * per_sm;
  const int grid = (int)(M < ctas ? M : ctas);
  return launch_pdl(kern, dim3(grid), 256, smem, stream, X, M, K, Q, S, status, limit_ns);
}

}  // namespace

int quant_launch(const void* X, bool x_bf16, int64_t M, int64_t K, bool to_e2m1, void* Q, void* S, int num_sms,
                 uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(X);
  const float* xf = static_cast<const float*>(X);
  uint8_t* q = static_cast<uint8_t*>(Q);
  if (!to_e2m1) {
    float* s = static_cast<float*>(S);
    const uint64_t row_bytes = (uint64_t)K * 4;
    if (!x_bf16 && row_bytes >= QS_MIN_ROW && row_bytes <= QS_MAX_ROW)
      return launch_staged(xf, M, K, q, s, num_sms, status, limit_ns, stream);
    const dim3 grid(grid_rows(M));
    if (x_bf16 && K <= QB_THREADS * QB_VPT * 8)
      return launch_pdl(quant_e4m3_rows_bf16_kernel<QB_THREADS, QB_VPT, QB_MINB>, grid, QB_THREADS, 0, stream, xb, M,
                        K, q, s);
    if (!x_bf16 && K <= 256 * 8 * 4) return launch_pdl(quant_e4m3_rows_f32_kernel, grid, 256, 0, stream, xf, M, K, q, s);
    if (x_bf16) return launch_pdl(quant_e4m3_rows_kernel<__nv_bfloat16>, grid, 256, 0, stream, xb, M, K, q, s);
    return launch_pdl(quant_e4m3_rows_kernel<float>, grid, 256, 0, stream, xf, M, K, q, s);
  }
  uint8_t* e = static_cast<uint8_t*>(S);
  const int rows = x_bf16 ? MxRows<__nv_bfloat16>::value : MxRows<float>::value;
  const int64_t groups = (M + rows - 1) / rows;
  const dim3 grid((unsigned)((K / 8 + 255) / 256), (unsigned)(groups < 65535 ? groups : 65535));
  if (x_bf16) return launch_pdl(quant_mxfp4_kernel<__nv_bfloat16>, grid, 256, 0, stream, xb, M, (int)K, q, e);
  return launch_pdl(quant_mxfp4_kernel<float>, grid, 256, 0, stream, xf, M, (int)K, q, e);
}

}  // namespace gp
