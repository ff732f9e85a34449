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
#include <cstdlib>

#include "kernels.h"
#include "ptx.cuh"

namespace gp {

constexpr int I8_CW = 8;  // warps per CTA, each with a private copy ring
constexpr int I8_THREADS = 32 * I8_CW;
// Two CTAs fit on one SM (registers <= 128/thread, shared memory <= 113 KiB),
// so with programmatic dependent launch the next GEMM's CTAs sit beside this
// one's and warm L2 with their weights while this one computes.
constexpr int I8_CTAS_PER_SM = 2;

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

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copy K tile `kt` (the 16 x 128-byte A tile and the strip's rows of the
// packed B tile) into a warp-private ring slot.  A rows >= M read as zeros.
// The A tile gets the 128-byte swizzle (chunk c of row r at slot c ^ (r%8));
// the packed B rows already carry it.
template <int SN>
__device__ __forceinline__ void i8_copy_ktile(const I8Params& p, const uint8_t* A, int mg, int n0, int rows, int kt,
                                              uint32_t slot, int lane) {
  const size_t kb = (size_t)p.ktiles * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = lane + 32 * j;
    const int row = i >> 3, c = i & 7;
    const int gm = mg * 16 + row;
    const bool valid = gm < p.M;
    cp_async_16(slot + row * 128 + ((c ^ (row & 7)) << 4), A + (size_t)(valid ? gm : 0) * kb + kt * 128 + c * 16,
                valid ? 16u : 0u);
  }
  const uint32_t sb = slot + 2048;
#pragma unroll 4
  for (int i = lane; i < rows * 8; i += 32) {
    const int row = i >> 3, c = i & 7;
    const int r = n0 + row;
    cp_async_16(sb + row * 128 + c * 16,
                p.Bp + (((size_t)(r >> 7) * p.ktiles + kt) * 128 + (r & 127)) * 128 + c * 16, 16u);
  }
}

template <int NB8, int R>
__global__ void __launch_bounds__(I8_THREADS, I8_CTAS_PER_SM) i8_gemm_kernel(const uint8_t* __restrict__ A, I8Params p) {
  constexpr int SN = NB8 * 8;
  constexpr int STAGE = 2048 + SN * 128;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * SN;
  const int rows = min(SN, p.N - n0);  // multiple of 16
  const int mg = blockIdx.y;
  const uint32_t ring = smem_u32(smem) + (uint32_t)(warp * R * STAGE);

  // Warm L2 with this warp's share of the weight strip while the previous
  // kernel on the stream may still run: a prefetch is only a cache hint.
  for (int kt = warp; kt < p.ktiles; kt += I8_CW) {
    if (lane == 0) {
      int r = n0;
      while (r < n0 + rows) {
        const int tn = r >> 7;
        const int r_end = min(n0 + rows, (tn + 1) << 7);
        prefetch_l2_bulk(p.Bp + ((size_t)tn * p.ktiles + kt) * 16384 + (size_t)(r & 127) * 128,
                         (uint32_t)(r_end - r) * 128u);
        r = r_end;
      }
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // A may be produced, and C read, by the previous kernel

  // Prologue: R K tiles of this warp in flight (one commit group each).
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int kt = warp + q * I8_CW;
    if (kt < p.ktiles) i8_copy_ktile<SN>(p, A, mg, n0, rows, kt, ring + q * STAGE, lane);
    cp_async_commit();
  }

  const int g = lane >> 2;  // mma group id: A rows g, g+8 and B row g of each 8-row block
  const int t = lane & 3;
  const int nb_valid = rows >> 3;
  int acc[NB8][4];
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0;

  int q = 0;
  for (int kt = warp; kt < p.ktiles; kt += I8_CW) {
    cp_async_wait<R - 1>();  // this lane's copies of the oldest tile are done
    __syncwarp();            // ... and every other lane's
    const uint8_t* sa = smem + (size_t)warp * R * STAGE + q * STAGE;
    const uint8_t* sbp = sa + 2048;
    const uint32_t slot_addr = ring + q * STAGE;
    const int kn = kt + R * I8_CW;
    q = (q + 1 == R) ? 0 : q + 1;
    float f[NB8][4];
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) f[nb][0] = f[nb][1] = f[nb][2] = f[nb][3] = 0.f;
    // Two 64-element halves of the K tile; only one half's raw bytes are live.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int slot = ((2 * t + h) ^ g) << 4;
      const uint4 ag = *reinterpret_cast<const uint4*>(sa + g * 128 + slot);
      const uint4 ag8 = *reinterpret_cast<const uint4*>(sa + (g + 8) * 128 + slot);
      uint4 bw[NB8];
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb)
        if (nb < nb_valid) bw[nb] = *reinterpret_cast<const uint4*>(sbp + (nb * 8 + g) * 128 + slot);
      if (h == 1) {
        __syncwarp();  // the slot is free: refill it with this warp's tile R steps ahead
        if (kn < p.ktiles) i8_copy_ktile<SN>(p, A, mg, n0, rows, kn, slot_addr, lane);
        cp_async_commit();
      }
      const uint32_t aw[4] = {ag.x, ag.y, ag.z, ag.w};
      const uint32_t a8w[4] = {ag8.x, ag8.y, ag8.z, ag8.w};
      uint32_t alo[4], ahi[4], a8lo[4], a8hi[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        i8x4_to_f16x2(aw[j], alo[j], ahi[j]);
        i8x4_to_f16x2(a8w[j], a8lo[j], a8hi[j]);
      }
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb) {
        if (nb < nb_valid) {
          const uint32_t w[4] = {bw[nb].x, bw[nb].y, bw[nb].z, bw[nb].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t blo, bhi;
            i8x4_to_f16x2(w[j], blo, bhi);
            mma_16816(f[nb], alo[j], a8lo[j], ahi[j], a8hi[j], blo, bhi);
          }
        }
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nb][i] += __float2int_rn(f[nb][i]);
    }
  }
  cp_async_wait<0>();

  // ------------------------------------------------------------ reduction
  __syncthreads();  // every warp is done with its ring
  int32_t* red = reinterpret_cast<int32_t*>(smem);  // [CW][16][SN]
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    const int col = nb * 8 + 2 * t;
    red[(warp * 16 + g) * SN + col] = acc[nb][0];
    red[(warp * 16 + g) * SN + col + 1] = acc[nb][1];
    red[(warp * 16 + g + 8) * SN + col] = acc[nb][2];
    red[(warp * 16 + g + 8) * SN + col + 1] = acc[nb][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * rows; i += I8_THREADS) {
    const int m = i / rows, n = i - m * rows;
    int sum = 0;
#pragma unroll
    for (int w = 0; w < I8_CW; ++w) sum += red[(w * 16 + m) * SN + n];
    const int gm = mg * 16 + m;
    if (gm < p.M) p.C[(size_t)gm * p.N + n0 + n] = sum;
  }
}

// Tuning overrides, read once per process: GP_I8_STRIP (rows of B per CTA:
// 16, 32, 48 or 64).
static int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  if (e == nullptr) return dflt;
  const int v = std::atoi(e);
  return v > 0 ? v : dflt;
}

template <int NB8, int R>
static int launch_i8(const uint8_t* A, I8Params p, dim3 grid, cudaStream_t stream) {
  constexpr int STAGE = 2048 + NB8 * 8 * 128;
  constexpr int RING = I8_CW * R * STAGE;
  constexpr int RED = I8_CW * 16 * NB8 * 8 * 4;
  constexpr int SMEM = RING > RED ? RING : RED;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  auto kern = i8_gemm_kernel<NB8, R>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
      return GP_ERR_CUDA;
    if (dev < 64) attr_set[dev] = true;
  }
  p.stages = R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(I8_THREADS);
  cfg.dynamicSmemBytes = (size_t)SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, A, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int i8_gemm_launch(const uint8_t* A, I8Params p, int num_sms, cudaStream_t stream) {
  // strip height: 16 * ceil(N / (16 * 2 * SMs)), at most 64 rows, so that
  // the strips fill both CTA slots of every SM
  static const int strip_override = env_int("GP_I8_STRIP", 0);
  const int slots = I8_CTAS_PER_SM * num_sms;
  int strip = 16 * ((p.N + 16 * slots - 1) / (16 * slots));
  if (strip_override == 16 || strip_override == 32 || strip_override == 48 || strip_override == 64)
    strip = strip_override;
  if (strip > 64) strip = 64;
  if (strip < 16) strip = 16;
  p.strip = strip;
  dim3 grid((unsigned)((p.N + strip - 1) / strip), (unsigned)((p.M + 15) / 16));
  switch (strip) {  // ring depth R per warp: R * 8 warps * stage bytes within shared memory
    case 16: return launch_i8<2, 2>(A, p, grid, stream);
    case 32: return launch_i8<4, 2>(A, p, grid, stream);
    case 48: return launch_i8<6, 1>(A, p, grid, stream);
    default: return launch_i8<8, 1>(A, p, grid, stream);
  }
}

}  // namespace gp
