// INT8 x INT8 -> INT32 GEMM for small M: weight streaming at HBM rate.
//
// "GEMM Optimization Guide", section 1.3: small batches (M <= 32) are
// memory-bound and want a large K tile for reuse.  Section 8.3: for
// M <= 512 the work is bandwidth, not MFMA, limited.  On GB300 the weight
// matrix B must stream from HBM once at full bandwidth:
//
//   - The grid is one wave.  Each CTA owns a strip of `strip` consecutive
//     rows of B (a multiple of 16, chosen so the strips roughly fill the
//     SMs) and all of K, for one group of 16 rows of A.  No split-K, so no
//     cross-CTA reduction.
//   - A producer warp (one lane) streams, per 128-byte K tile:
//       * the 16 x 128-byte A tile (2-D TMA, 128-byte swizzle, rows >= M
//         zero-filled);
//       * the strip's packed-B rows, as one or two contiguous bulk copies
//         (the packed layout keeps each 128-row band's K tile contiguous).
//     These go into a deep ring of stages (up to 192 KiB in flight per SM),
//     with full/empty mbarriers.
//   - Eight consumer warps take K tiles round-robin.  sm_103a has no
//     tcgen05 integer MMA and its int8 tensor and dp4a rates (~150 TOPS
//     measured) cannot keep pace with the weight stream, so the consumers
//     use the 16-bit MMA:
//       * int8 values are exact in fp16;
//       * products are exact;
//       * a 128-element K tile sums to at most 128 * 128 * 128 = 2^21 in
//         magnitude, so its fp32 accumulation is exact;
//       * each K tile's fp32 partials are converted to int32 and added in
//         int32.
//     The result is the exact integer product.  The int8 -> fp16
//     conversion is 5 integer/half ops per 4 values (xor, 2 byte permutes,
//     2 packed subtracts of the 1024+128 bias).
//   - K is permuted identically for A and B inside each 64-element group,
//     which leaves the sum unchanged.  Lane t reads bytes
//     [32t, 32t+32) of a row.  Those bytes sit in 16-byte slots
//     (2t+h) ^ (row % 8), so the 8 lanes of each shared-memory phase hit
//     8 distinct bank groups.
//   - The 8 warps' int32 partials are reduced through shared memory and
//     stored as coalesced int32 rows of C.
#include "kernels.h"
#include "ptx.cuh"

namespace gp {

constexpr int I8_CW = 8;                     // consumer warps
constexpr int I8_THREADS = 32 * (I8_CW + 1);  // + one producer warp
constexpr int I8_RING_BUDGET = 192 * 1024;

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

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NB8>
__global__ void __launch_bounds__(I8_THREADS, 1) i8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, I8Params p) {
  constexpr int SN = NB8 * 8;
  constexpr int STAGE = 2048 + SN * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  const int ring = stages * STAGE;
  const int red_bytes = I8_CW * 16 * SN * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (ring > red_bytes ? ring : red_bytes));
  uint64_t* empty = full + stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + stages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * SN;
  const int rows = min(SN, p.N - n0);  // multiple of 16
  const int mg = blockIdx.y;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
  }
  __syncthreads();

  if (warp == I8_CW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_b = policy_evict_first();
      uint32_t issued = 0;
      bool ok = true;
      for (int kt = 0; kt < p.ktiles; ++kt) {
        const int s = kt % stages;
        const uint32_t ph = (uint32_t)(kt / stages) & 1;
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        uint8_t* st = base + s * STAGE;
        mbar_arrive_expect_tx(&full[s], 2048u + (uint32_t)rows * 128u);
        tma_load_2d(st, &tmA, kt * 128, mg * 16, &full[s]);
        int r = n0;
        while (r < n0 + rows) {
          const int tn = r >> 7;
          const int r_end = min(n0 + rows, (tn + 1) << 7);
          bulk_load_hint(st + 2048 + (r - n0) * 128,
                         p.Bp + ((size_t)tn * p.ktiles + kt) * 16384 + (size_t)(r & 127) * 128,
                         (uint32_t)(r_end - r) * 128u, &full[s], pol_b);
          r = r_end;
        }
        ++issued;
      }
      if (!ok) {
        const uint32_t n = issued < (uint32_t)stages ? issued : (uint32_t)stages;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t q = issued - 1 - i;
          volatile int never = 0;
          wait_bounded(&full[q % stages], (q / stages) & 1, &never, p.status, ST_TIMEOUT_DRAIN, p.wait_limit_ns);
        }
      }
    }
    return;  // the producer takes no part in the reduction below
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2;  // mma group id: A rows g, g+8 and B row g of each 8-row block
  const int t = lane & 3;
  const int nb_valid = rows >> 3;
  int acc[NB8][4];
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0;

  for (int kt = warp; kt < p.ktiles; kt += I8_CW) {
    const int s = kt % stages;
    const uint32_t ph = (uint32_t)(kt / stages) & 1;
    if (!wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_CONSUMER, p.wait_limit_ns)) break;
    const uint32_t sa = smem_u32(base + s * STAGE);
    const uint32_t sb = sa + 2048;
    float f[NB8][4];
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) f[nb][0] = f[nb][1] = f[nb][2] = f[nb][3] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t slot = (uint32_t)(((2 * t + h) ^ g) << 4);
      uint32_t ag[4], ag8[4];
      ld_shared_v4(sa + g * 128 + slot, ag[0], ag[1], ag[2], ag[3]);
      ld_shared_v4(sa + (g + 8) * 128 + slot, ag8[0], ag8[1], ag8[2], ag8[3]);
      uint32_t alo[4], ahi[4], a8lo[4], a8hi[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        i8x4_to_f16x2(ag[j], alo[j], ahi[j]);
        i8x4_to_f16x2(ag8[j], a8lo[j], a8hi[j]);
      }
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb) {
        if (nb < nb_valid) {
          uint32_t bw[4];
          ld_shared_v4(sb + (nb * 8 + g) * 128 + slot, bw[0], bw[1], bw[2], bw[3]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t blo, bhi;
            i8x4_to_f16x2(bw[j], blo, bhi);
            mma_16816(f[nb], alo[j], a8lo[j], ahi[j], a8hi[j], blo, bhi);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nb][i] += __float2int_rn(f[nb][i]);
    }
  }

  // ------------------------------------------------------------ reduction
  named_bar_sync(1, I8_CW * 32);  // every consumer is done with the ring
  int32_t* red = reinterpret_cast<int32_t*>(base);  // [CW][16][SN]
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    const int col = nb * 8 + 2 * t;
    red[(warp * 16 + g) * SN + col] = acc[nb][0];
    red[(warp * 16 + g) * SN + col + 1] = acc[nb][1];
    red[(warp * 16 + g + 8) * SN + col] = acc[nb][2];
    red[(warp * 16 + g + 8) * SN + col + 1] = acc[nb][3];
  }
  named_bar_sync(1, I8_CW * 32);
  for (int i = threadIdx.x; i < 16 * rows; i += I8_CW * 32) {
    const int m = i / rows, n = i - m * rows;
    int sum = 0;
#pragma unroll
    for (int w = 0; w < I8_CW; ++w) sum += red[(w * 16 + m) * SN + n];
    const int gm = mg * 16 + m;
    if (gm < p.M) p.C[(size_t)gm * p.N + n0 + n] = sum;
  }
}

template <int NB8>
static int launch_i8(const CUtensorMap& tmA, I8Params p, dim3 grid, cudaStream_t stream) {
  constexpr int STAGE = 2048 + NB8 * 8 * 128;
  int stages = I8_RING_BUDGET / STAGE;
  if (stages > p.ktiles) stages = p.ktiles;
  if (stages < 1) stages = 1;
  p.stages = stages;
  const int ring = stages * STAGE;
  const int red = I8_CW * 16 * NB8 * 8 * 4;
  const int smem = (ring > red ? ring : red) + 2 * stages * 8 + 16 + 1024;
  auto kern = i8_gemm_kernel<NB8>;
  // the attribute is set once per device to the largest size this launcher uses
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev]) {
    const int max_smem = (I8_RING_BUDGET > I8_CW * 16 * 64 * 4 ? I8_RING_BUDGET : I8_CW * 16 * 64 * 4) + 2 * 256 * 8 +
                         16 + 1024;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess)
      return GP_ERR_CUDA;
    if (dev < 64) attr_set[dev] = true;
  }
  kern<<<grid, I8_THREADS, smem, stream>>>(tmA, p);
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int i8_gemm_launch(const CUtensorMap& tmA, I8Params p, int num_sms, cudaStream_t stream) {
  // strip height: 16 * ceil(N / (16 * SMs)), at most 64 rows
  int strip = 16 * ((p.N + 16 * num_sms - 1) / (16 * num_sms));
  if (strip > 64) strip = 64;
  if (strip < 16) strip = 16;
  p.strip = strip;
  dim3 grid((unsigned)((p.N + strip - 1) / strip), (unsigned)((p.M + 15) / 16));
  switch (strip) {
    case 16: return launch_i8<2>(tmA, p, grid, stream);
    case 32: return launch_i8<4>(tmA, p, grid, stream);
    case 48: return launch_i8<6>(tmA, p, grid, stream);
    default: return launch_i8<8>(tmA, p, grid, stream);
  }
}

}  // namespace gp
