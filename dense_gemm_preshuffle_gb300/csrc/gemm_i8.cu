// INT8 x INT8 -> INT32 GEMM for small M: weight streaming at HBM rate.
//
// "GEMM Optimization Guide", section 1.3: small batches (M <= 32) are
// memory-bound and want a large K tile for reuse.  Section 8.3: for
// M <= 512 the work is bandwidth, not MFMA, limited.  On GB300 the weight
// matrix B must stream from HBM once at full bandwidth:
//
//   - The grid is one wave.  Each CTA owns a strip of `strip` consecutive
//     rows of B (a multiple of 16, chosen so that two strips share an SM
//     where N allows) and all of K, for one group of 16 rows of A.  The
//     INT8 packed layout stores 8-row bands, so a strip's rows for 8 K tiles
//     are one 4-D TMA box.
//   - Narrow N (fewer strips than SMs): the strip's K stages are split over
//     the 2, 4 or 8 CTAs of a thread-block cluster.  Each rank streams its
//     range of B and A; the int32 partials (each with its own offset
//     correction) are summed exactly through distributed shared memory,
//     every rank storing a slice of the strip's columns.
//   - A CTA takes under half of an SM, so with programmatic dependent
//     launch the next GEMM's CTAs start beside this one's on the SMs that
//     hold a single strip: they warm L2 with their weights and, for constant
//     weights (GP_RUN_B_CONSTANT), fill their ring with B before the wait on
//     this kernel.
//   - One producer warp.  Each thread's bulk copies complete one after
//     another, so every copy of a stage has its own lane: INT8 B as one
//     plain bulk copy per 8-row unit (the unit's 8 K tiles are adjacent in
//     the packed layout), W4A8 B as one TMA box, and A from the next lane.
//     Stages of 8 K tiles (up to 48 KiB) go into a ring of 2, with
//     full/empty mbarriers.
//   - Eight consumer warps; warp w computes K tile w of every stage.  sm_103a
//     has no tcgen05 integer MMA and its int8 tensor and dp4a rates (~150
//     TOPS measured) cannot keep pace with the weight stream, so the
//     consumers use the 16-bit MMA on exact fp16 images of the integers:
//       * A (row-major int8 from the caller): a -> fp16 a, 5 integer/half
//         ops per 4 values (xor, 2 byte permutes into the 0x64XX binade,
//         2 packed subtracts of 1024 + 128);
//       * B (packed offline in offset binary, byte u = b + 128): u -> the
//         fp16 subnormal u * 2^-24, 2 byte permutes per 4 values and no
//         arithmetic;
//       * products a * u * 2^-24 are exact, and a 128-element K tile sums
//         to |sum a*u| <= 128 * 128 * 255 < 2^22 units of 2^-24, so its
//         fp32 accumulation is exact;
//       * each K tile's partials are scaled back to integers with one FMA
//         (x * 2^24 + 1.5 * 2^23 is exact and holds x in its low bits) and
//         added in int32;
//       * sum a*b = sum a*u - 128 * sum a, with the row sums of A taken by
//         dp4a from the same A words.
//     The result is the exact integer product.
//   - K is permuted identically for A and B inside each 64-element group,
//     which leaves the sum unchanged.  Lane t reads bytes
//     [32t, 32t+32) of a row.  Those bytes sit in 16-byte slots
//     (2t+h) ^ (row % 8), so the 8 lanes of each shared-memory phase hit
//     8 distinct bank groups.
//   - The 8 warps' int32 partials are reduced through shared memory and
//     stored as coalesced int32 rows of C.
#include <cstdlib>

#include "i8_math.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace gp {

constexpr int I8_CW = 8;                 // consumer warps 0..7
constexpr int I8_PRODUCER = I8_CW;       // warp 8: lane 0 issues B, lane 1 issues A
constexpr int I8_THREADS = 32 * (I8_CW + 1);
constexpr int I8_KT = I8_CW;             // K tiles per stage: one per consumer warp
constexpr int I8_STAGES = 2;
// Two CTAs share an SM for strips of up to 32 rows (three for 16 rows).
constexpr int I8_CTAS_PER_SM = 2;
__host__ __device__ constexpr int i8_ctas_per_sm(int nb8) { return nb8 <= 2 ? 3 : (nb8 <= 4 ? 2 : 1); }

// NB8: eight-row units per strip.  W4: B is W4A8's int4 (a packed 128-byte
// B tile then spans two 128-element K tiles of A).  SPLIT: CTAs of a
// thread-block cluster that share one strip, each over a contiguous range of
// its K stages (1: no split).
template <int NB8, bool W4, int SPLIT>
__global__ void __launch_bounds__(I8_THREADS, i8_ctas_per_sm(NB8))
    i8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, I8Params p) {
  static_assert(SPLIT == 1 || SPLIT == 2 || SPLIT == 4 || SPLIT == 8, "cluster sizes of the K split");
  constexpr int SN = NB8 * 8;                    // rows of B per CTA
  constexpr int BT = W4 ? I8_KT / 2 : I8_KT;     // packed B tiles (128 B per row) per stage
  constexpr int A_BYTES = I8_KT * 16 * 128;      // [kt][16 rows][128 B], 128-byte swizzle
  constexpr int B_BYTES = BT * SN * 128;         // [unit][B tile][8 rows][128 B], packed swizzle
  constexpr int STAGE = A_BYTES + B_BYTES;
  // K split: this CTA's int32 partial [16][SN], after the ring's barriers
  constexpr int PART_OFF = I8_STAGES * STAGE + 64;
  constexpr int PART_BYTES = SPLIT > 1 ? 16 * SN * 4 : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + I8_STAGES * STAGE);
  uint64_t* empty = full + I8_STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + I8_STAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int units = p.N >> 3;
  // K split: the SPLIT CTAs of a cluster share strip blockIdx.x / SPLIT, and
  // rank r takes K stages [q0, q1) of the strip's nst (all of them, and
  // rank 0, without a split).
  const uint32_t rank = SPLIT > 1 ? cluster_ctarank() : 0u;
  const int u0 = ((int)blockIdx.x / SPLIT) * NB8;
  const int nu = min(NB8, units - u0);  // units of this strip that exist (the last strip may be short)
  const int mg = p.mg0 + (int)blockIdx.y;  // this CTA's group of 16 rows of A
  const int nst = (p.ktiles + I8_KT - 1) / I8_KT;
  const int q0 = (int)rank * nst / SPLIT;
  const int nstages = ((int)rank + 1) * nst / SPLIT - q0;  // this CTA's stages, q0 + [0, nstages)
  const uint64_t limit = p.wait_limit_ns;
  {
    // Launch self-check (uniform over the CTA, and over its cluster, before
    // any copy): the strip exists, the rows of A exist, every rank of the
    // split has a stage, the cluster has SPLIT CTAs, and the ring fits the
    // dynamic shared memory.  A mismatch is recorded and the CTA returns;
    // the whole cluster then returns, so no CTA is left at a cluster barrier.
    uint32_t dyn, ncta = 1;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if constexpr (SPLIT > 1) asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    const uint32_t need = SPLIT > 1 ? (uint32_t)(base + PART_OFF + PART_BYTES - smem_raw)
                                     : (uint32_t)(reinterpret_cast<const volatile uint8_t*>(abort_flag + 1) - smem_raw);
    if (nu < 1 || mg * 16 >= p.M || p.ktiles < 1 || nst < SPLIT || ncta != (uint32_t)SPLIT || need > dyn ||
        (int)blockDim.x != I8_THREADS) {
      if (threadIdx.x == 0) atomicOr(p.status, ST_BAD_LAUNCH);
      pdl_wait();  // complete after the previous kernel all the same
      return;
    }
  }

  // B issuers: INT8 B travels as one plain bulk copy per 8-row unit (its K
  // tiles are adjacent in the packed layout), each issued by the unit's own
  // producer lane, since one thread's bulk copies complete one after
  // another; W4A8's B (half the bytes) as one 4-D TMA box.  The A issuer is
  // the next lane.
  constexpr int B_ISSUERS = W4 ? 1 : NB8;
  static_assert(B_ISSUERS + 1 <= 32, "one producer lane per copy");
  if (threadIdx.x == 0) {
    for (int s = 0; s < I8_STAGES; ++s) {
      mbar_init(&full[s], B_ISSUERS + 1);  // the B issuers and the A issuer
      mbar_init(&empty[s], I8_CW);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  // B for stage q from issuer lane `bl`.  INT8: unit u0 + bl, its K tiles
  // [8q, 8q + 8) (fewer at the end of K), one contiguous run; a unit past N
  // or K tiles past the end are not read, and the consumers never use their
  // bytes.  W4A8: NB8 units x BT packed tiles of 8 rows in one TMA box, units
  // past N read as zeros.
  auto load_b = [&](int lq, int bl) {
    const int s = lq % I8_STAGES;
    const int q = q0 + lq;
    if constexpr (!W4) {
      const int u = u0 + bl;
      const int kt0 = q * I8_KT;
      const int nkt = min(I8_KT, p.ktiles - kt0);
      const uint32_t bytes = (u < units && nkt > 0) ? (uint32_t)nkt * 1024u : 0u;
      mbar_arrive_expect_tx(&full[s], bytes);
      if (bytes != 0)
        bulk_load(base + s * STAGE + A_BYTES + bl * (I8_KT * 8 * 128), p.Bp + ((size_t)u * p.ktiles + kt0) * 1024,
                  bytes, &full[s]);
      return;
    }
    mbar_arrive_expect_tx(&full[s], B_BYTES);
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::
            "r"(smem_u32(base + s * STAGE + A_BYTES)),
        "l"(reinterpret_cast<uint64_t>(&tmB)), "r"(0), "r"(0), "r"(q * BT), "r"(u0), "r"(smem_u32(&full[s]))
        : "memory");
  };
  // A: I8_KT K tiles x 16 rows x 128 B (rows >= M and K tiles >= ktiles read as zeros)
  auto load_a = [&](int lq) {
    const int s = lq % I8_STAGES;
    const int q = q0 + lq;
    mbar_arrive_expect_tx(&full[s], A_BYTES);
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_u32(base + s * STAGE)),
        "l"(reinterpret_cast<uint64_t>(&tmA)), "r"(0), "r"(mg * 16), "r"(q * I8_KT), "r"(smem_u32(&full[s]))
        : "memory");
  };
  // With constant weights the ring's first stages of B are requested before
  // the wait on the previous kernel; the rest of the strip is warmed in L2.
  // An independent call (which implies constant weights) does not wait
  // here at all: its whole body runs alongside the previous kernel, and it
  // waits for that kernel at exit.
  const int early = p.b_constant ? min(nstages, I8_STAGES) : 0;
  if (threadIdx.x == I8_PRODUCER * 32) {
    // A prefetch is only a cache hint: safe while the previous kernel runs.
    for (int q = q0 + early; q < q0 + nstages; ++q)
      asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                       reinterpret_cast<uint64_t>(&tmB)),
                   "r"(0), "r"(0), "r"(q * BT), "r"(u0)
                   : "memory");
  }
  if (threadIdx.x == 32) {
    // A is warmed in L2 too (the previous kernel may still write it; L2
    // stays coherent, so the hint is harmless).
    for (int q = q0; q < q0 + nstages; ++q)
      asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                       reinterpret_cast<uint64_t>(&tmA)),
                   "r"(0), "r"(mg * 16), "r"(q * I8_KT)
                   : "memory");
  }
  pdl_launch_dependents();
  __syncthreads();
  // Fault injection (host-selected): B is issued only up to, not including,
  // stage debug_skip_load - 1, so the consumers' waits on that stage must
  // time out. The bound is computed once, off the per-stage path.
  const int b_end = p.debug_skip_load > 0 ? min(nstages, p.debug_skip_load - 1) : nstages;
  if (warp == I8_PRODUCER && lane < B_ISSUERS)
    for (int q = 0; q < min(early, b_end); ++q) load_b(q, lane);
  if (!p.independent) pdl_wait();  // A may be produced, and C read, by the previous kernel

  if (warp == I8_PRODUCER) {
    // ------------------------------------------------------------ producers
    if (lane <= B_ISSUERS) {
      const bool is_b = lane < B_ISSUERS;
      int q = is_b ? min(early, b_end) : 0;
      const int q_end = is_b ? b_end : nstages;
      bool ok = true;
      for (; q < q_end; ++q) {
        const int s = q % I8_STAGES;
        const uint32_t ph = (uint32_t)(q / I8_STAGES) & 1;
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
          ok = false;
          break;
        }
        if (is_b)
          load_b(q, lane);
        else
          load_a(q);
      }
      if (!ok || *abort_flag) {
        // wait (bounded) for this thread's copies still in flight
        const int issued = q;
        for (int i = 0; i < I8_STAGES && i < issued; ++i) {
          const int qq = issued - 1 - i;
          volatile int never = 0;
          wait_bounded(&full[qq % I8_STAGES], (uint32_t)(qq / I8_STAGES) & 1, &never, p.status, ST_TIMEOUT_DRAIN,
                       limit);
        }
      }
    }
    if constexpr (SPLIT > 1) {
      // the producer takes no part in the reduction below, but every thread
      // of the cluster passes both of its cluster barriers
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  // Every warp sees every stage (warp w takes K tile w), so each waits on
  // consecutive phases of every barrier.
  const int g = lane >> 2;  // mma group id: A rows g, g+8 and row g of each 8-row unit
  const int t = lane & 3;
  int acc[NB8][4];
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0;
  int rs_lo = 0, rs_hi = 0;  // this lane's share of the row sums of A rows g and g + 8

  for (int q = 0; q < nstages; ++q) {
    const int s = q % I8_STAGES;
    const uint32_t ph = (uint32_t)(q / I8_STAGES) & 1;
    if (!wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_CONSUMER, limit)) break;
    const bool live = (q0 + q) * I8_KT + warp < p.ktiles;
    const uint8_t* sa = base + s * STAGE + warp * (16 * 128);
    float f[NB8][4];
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) f[nb][0] = f[nb][1] = f[nb][2] = f[nb][3] = 0.f;
    if constexpr (W4) {
      // K tile `warp` of A is half of packed B tile warp / 2: lane t's 32 K
      // values are one 16-byte chunk, 4 * (warp % 2) + t, of each B row,
      // stored at slot chunk ^ g ^ 4 (g % 2) (the W4A8 packing), so the 8
      // lanes of rows g and g ^ 1 that load together hit 8 distinct bank
      // groups.
      const uint8_t* sb = base + s * STAGE + A_BYTES + ((warp >> 1) * 8 + g) * 128 +
                          (((4 * (warp & 1) + t) ^ g ^ ((g & 1) << 2)) << 4);  // + unit * (BT * 8 * 128)
      uint4 bw[NB8];
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb) bw[nb] = *reinterpret_cast<const uint4*>(sb + nb * (BT * 8 * 128));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int slot = ((2 * t + h) ^ g) << 4;
        const uint4 ag = *reinterpret_cast<const uint4*>(sa + g * 128 + slot);
        const uint4 ag8 = *reinterpret_cast<const uint4*>(sa + (g + 8) * 128 + slot);
        if (h == 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);  // this warp's reads of the stage are done
        }
        if (live) {
          const uint32_t aw[4] = {ag.x, ag.y, ag.z, ag.w};
          const uint32_t a8w[4] = {ag8.x, ag8.y, ag8.z, ag8.w};
          uint32_t alo[4], ahi[4], a8lo[4], a8hi[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            i8x4_to_f16x2(aw[j], alo[j], ahi[j]);
            i8x4_to_f16x2(a8w[j], a8lo[j], a8hi[j]);
            rs_lo = __dp4a((int)aw[j], 0x01010101, rs_lo);
            rs_hi = __dp4a((int)a8w[j], 0x01010101, rs_hi);
          }
          // Units innermost: consecutive MMAs use different accumulators, so
          // their latencies overlap.  Units past N (zeros from the TMA box)
          // are computed too and never stored.
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb) {
              // A word j holds K values 4j..4j+3 of this half: B word j / 2,
              // nibble pairs (0,1),(2,3) or (4,5),(6,7) as fp16 subnormals
              const uint32_t w = (h == 0 ? (j < 2 ? bw[nb].x : bw[nb].y) : (j < 2 ? bw[nb].z : bw[nb].w)) >>
                                 ((j & 1) * 8);
              mma_16816(f[nb], alo[j], a8lo[j], ahi[j], a8hi[j], w & 0x000F000Fu, (w >> 4) & 0x000F000Fu);
            }
          }
        }
      }
    } else {
      const uint8_t* sb = base + s * STAGE + A_BYTES + (warp * 8 + g) * 128;  // + unit * (I8_KT * 8 * 128)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int slot = ((2 * t + h) ^ g) << 4;
        const uint4 ag = *reinterpret_cast<const uint4*>(sa + g * 128 + slot);
        const uint4 ag8 = *reinterpret_cast<const uint4*>(sa + (g + 8) * 128 + slot);
        uint4 bw[NB8];
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb)
          bw[nb] = *reinterpret_cast<const uint4*>(sb + nb * (I8_KT * 8 * 128) + slot);
        if (h == 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);  // this warp's reads of the stage are done
        }
        if (live) {
          const uint32_t aw[4] = {ag.x, ag.y, ag.z, ag.w};
          const uint32_t a8w[4] = {ag8.x, ag8.y, ag8.z, ag8.w};
          uint32_t alo[4], ahi[4], a8lo[4], a8hi[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            i8x4_to_f16x2(aw[j], alo[j], ahi[j]);
            i8x4_to_f16x2(a8w[j], a8lo[j], a8hi[j]);
            rs_lo = __dp4a((int)aw[j], 0x01010101, rs_lo);
            rs_hi = __dp4a((int)a8w[j], 0x01010101, rs_hi);
          }
          // Units innermost: consecutive MMAs use different accumulators, so
          // their latencies overlap.  Units past N (zeros from the TMA box)
          // are computed too and never stored.
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb) {
              const uint32_t w = j == 0 ? bw[nb].x : j == 1 ? bw[nb].y : j == 2 ? bw[nb].z : bw[nb].w;
              uint32_t blo, bhi;
              u8x4_to_f16x2_sub(w, blo, bhi);
              mma_16816(f[nb], alo[j], a8lo[j], ahi[j], a8hi[j], blo, bhi);
            }
          }
        }
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nb][i] += scaled_to_int(f[nb][i]);
    }
  }
  // full row sums over this warp's K tiles (the 4 lanes of a group hold
  // disjoint 32-byte slices of every K tile)
  rs_lo += __shfl_xor_sync(0xffffffffu, rs_lo, 1);
  rs_lo += __shfl_xor_sync(0xffffffffu, rs_lo, 2);
  rs_hi += __shfl_xor_sync(0xffffffffu, rs_hi, 1);
  rs_hi += __shfl_xor_sync(0xffffffffu, rs_hi, 2);

  // ------------------------------------------------------------ reduction
  named_bar_sync(1, I8_CW * 32);  // every consumer is done with the ring (no copy in flight)
  // [CW][16][RS] partials.  A lane stores its two adjacent columns as one
  // 8-byte word; with the row stride RS = 8 (mod 32) ints, the 16 lanes of
  // each half-warp (rows g, 4 column pairs each) hit 16 distinct bank pairs
  // (a stride of 32 put all 8 rows on the same banks: 8-way conflicts).
  constexpr int RS = ((SN - 8 + 31) / 32) * 32 + 8;
  static_assert(I8_CW * 16 * RS * 4 <= I8_STAGES * STAGE, "the reduction fits in the ring");
  int32_t* red = reinterpret_cast<int32_t*>(base);
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    const int col = nb * 8 + 2 * t;
    // sum a*b = sum a*(b + bias) - bias * sum a (bias 128 for int8 B, 8 for int4)
    constexpr int OFF = W4 ? 8 : 128;
    *reinterpret_cast<int2*>(red + (warp * 16 + g) * RS + col) =
        make_int2(acc[nb][0] - OFF * rs_lo, acc[nb][1] - OFF * rs_lo);
    *reinterpret_cast<int2*>(red + (warp * 16 + g + 8) * RS + col) =
        make_int2(acc[nb][2] - OFF * rs_hi, acc[nb][3] - OFF * rs_hi);
  }
  named_bar_sync(1, I8_CW * 32);
  const int cols = nu * 8;
  const int n0 = u0 * 8;
  if constexpr (SPLIT == 1) {
    for (int i = threadIdx.x; i < 16 * cols; i += I8_CW * 32) {
      const int m = i / cols, n = i - m * cols;
      int sum = 0;
#pragma unroll
      for (int w = 0; w < I8_CW; ++w) sum += red[(w * 16 + m) * RS + n];
      const int gm = mg * 16 + m;
      if (gm < p.M) p.C[(size_t)gm * p.N + n0 + n] = sum;
    }
  } else {
    // K split: this CTA's partial [16][SN] goes to its own buffer beside the
    // ring; after a cluster barrier (release / acquire) rank r sums columns
    // [r cols / SPLIT, (r + 1) cols / SPLIT) of every rank's partial, read
    // through distributed shared memory in rank order, and stores them.
    // Integer sums: exact in any order.  A second cluster barrier keeps
    // every partial alive until its last remote read.
    int32_t* part = reinterpret_cast<int32_t*>(base + PART_OFF);
    for (int i = threadIdx.x; i < 16 * cols; i += I8_CW * 32) {
      const int m = i / cols, n = i - m * cols;
      int sum = 0;
#pragma unroll
      for (int w = 0; w < I8_CW; ++w) sum += red[(w * 16 + m) * RS + n];
      part[m * SN + n] = sum;
    }
    cluster_sync_all();
    const int c0 = (int)rank * cols / SPLIT;
    const int nc = ((int)rank + 1) * cols / SPLIT - c0;
    for (int i = threadIdx.x; i < 16 * nc; i += I8_CW * 32) {
      const int m = i / nc, n = c0 + (i - m * nc);
      const uint32_t addr = smem_u32(part + m * SN + n);
      int sum = 0;
#pragma unroll
      for (int j = 0; j < SPLIT; ++j) sum += (int)ld_shared_cluster_u32(mapa_shared(addr, (uint32_t)j));
      const int gm = mg * 16 + m;
      if (gm < p.M) p.C[(size_t)gm * p.N + n0 + n] = sum;
    }
    cluster_sync_all();
  }
  // An independent call completes only after the kernel before it, so a
  // later kernel's wait on this one covers everything earlier on the stream.
  if (p.independent) pdl_wait();
}

// Tuning overrides, read once per process: GP_I8_STRIP (rows of B per CTA:
// 16, 24, 32, 48 or 64) and GP_I8_SPLITK (1, 2, 4 or 8).
static int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  if (e == nullptr) return dflt;
  const int v = std::atoi(e);
  return v > 0 ? v : dflt;
}

template <int NB8, bool W4, int SPLIT = 1>
static int launch_i8(const CUtensorMap& tmA, const CUtensorMap& tmB, I8Params p, dim3 grid, cudaStream_t stream) {
  constexpr int STAGE = I8_KT * 16 * 128 + (W4 ? I8_KT / 2 : I8_KT) * NB8 * 8 * 128;
  constexpr int RED = I8_CW * 16 * NB8 * 8 * 4;
  constexpr int RING = I8_STAGES * STAGE;
  static_assert(RED <= RING, "the reduction reuses the ring");
  // the ring, its barriers (64 bytes), the K split's partial, alignment slack
  constexpr int SMEM = RING + 64 + (SPLIT > 1 ? 16 * NB8 * 8 * 4 : 0) + 1024;
  static_assert(SMEM * i8_ctas_per_sm(NB8) <= 228 * 1024, "shared memory budget");
  auto kern = i8_gemm_kernel<NB8, W4, SPLIT>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, SMEM); rc != GP_OK) return rc;
  p.stages = I8_STAGES;
  grid.x *= SPLIT;  // SPLIT consecutive CTAs, one cluster, per strip
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(I8_THREADS);
  cfg.dynamicSmemBytes = (size_t)SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = SPLIT;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = SPLIT > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int i8_strip_rows(int N, int num_sms) {
  // Rows of B per CTA, a multiple of 16.  Prefer strips of at most 32 rows,
  // which let two CTAs share an SM: with programmatic dependent launch the
  // next product's CTAs then sit beside this one's and stream while it
  // computes (measured 8.5 us against 9.5 us for one 48-row strip per SM at
  // 16 x 7168 x 4096).  Wider problems take one strip per SM, at most 64
  // rows.  GP_I8_STRIP (16, 24, 32, 48 or 64) overrides.
  static const int strip_override = env_int("GP_I8_STRIP", 0);
  if (strip_override == 16 || strip_override == 24 || strip_override == 32 || strip_override == 48 ||
      strip_override == 64)
    return strip_override;
  const int two_per_sm = 16 * ((N + 16 * I8_CTAS_PER_SM * num_sms - 1) / (16 * I8_CTAS_PER_SM * num_sms));
  if (two_per_sm <= 32) return two_per_sm;
  const int one_per_sm = 16 * ((N + 16 * num_sms - 1) / (16 * num_sms));
  return one_per_sm > 64 ? 64 : one_per_sm;
}

static int i8_gemm_launch_groups(const CUtensorMap& tmA, const CUtensorMap& tmB, I8Params p, int ngroups,
                                 cudaStream_t stream);

int i8_gemm_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, I8Params p, int num_sms, cudaStream_t stream) {
  const int groups = (p.M + 15) / 16;  // groups of 16 rows of A
  if (groups > 65535) {
    // more row groups than one grid's y extent: one launch per 65535 groups
    for (int g0 = 0; g0 < groups; g0 += 65535) {
      I8Params q = p;
      q.mg0 = g0;
      const int rc = i8_gemm_launch_groups(tmA, tmB, q, min(65535, groups - g0), stream);
      if (rc != GP_OK) return rc;
    }
    return GP_OK;
  }
  p.mg0 = 0;
  return i8_gemm_launch_groups(tmA, tmB, p, groups, stream);
}

int i8_split_k(int64_t ctas, int ktiles, int strip, int num_sms) {
  // K split over a cluster for products whose strips alone leave SMs
  // without a CTA (narrow N): the largest split in {2, 4, 8} that keeps the
  // grid within one wave of resident CTAs and gives every rank at least two
  // stages of 8 K tiles, so that each CTA's two-stage ring still overlaps
  // its copies with its MMAs.  Built for 16- and 32-row strips (a split of
  // 8, the portable cluster limit, for 16-row strips only).
  // GP_I8_SPLITK (1, 2, 4 or 8) forces a split where it is valid, for sweeps.
  static const int forced = env_int("GP_I8_SPLITK", 0);
  const int nst = (ktiles + I8_KT - 1) / I8_KT;
  if (strip != 16 && strip != 32) return 1;
  auto built = [&](int s) { return s != 8 || strip == 16; };
  if (forced == 1 || forced == 2 || forced == 4 || forced == 8) return (nst >= forced && built(forced)) ? forced : 1;
  if (ctas >= num_sms) return 1;
  const int64_t slots = (int64_t)num_sms * i8_ctas_per_sm(strip / 8);
  int split = 1;
  for (int s : {2, 4, 8})
    if (built(s) && ctas * s <= slots && nst >= 2 * s) split = s;
  return split;
}

static int i8_gemm_launch_groups(const CUtensorMap& tmA, const CUtensorMap& tmB, I8Params p, int ngroups,
                                 cudaStream_t stream) {
  const int strip = p.strip;
  dim3 grid((unsigned)((p.N + strip - 1) / strip), (unsigned)ngroups);
  const int split = p.split;
  if (split == 8) {
    // 16-row strips only (i8_split_k)
    if (strip != 16) return GP_ERR_UNSUPPORTED;
    return p.w4 ? launch_i8<2, true, 8>(tmA, tmB, p, grid, stream) : launch_i8<2, false, 8>(tmA, tmB, p, grid, stream);
  }
  if (split == 2 || split == 4) {
    // strips of 16 or 32 rows only (i8_split_k)
    if (strip == 16) {
      if (p.w4) return split == 2 ? launch_i8<2, true, 2>(tmA, tmB, p, grid, stream)
                                  : launch_i8<2, true, 4>(tmA, tmB, p, grid, stream);
      return split == 2 ? launch_i8<2, false, 2>(tmA, tmB, p, grid, stream)
                        : launch_i8<2, false, 4>(tmA, tmB, p, grid, stream);
    }
    if (strip == 32) {
      if (p.w4) return split == 2 ? launch_i8<4, true, 2>(tmA, tmB, p, grid, stream)
                                  : launch_i8<4, true, 4>(tmA, tmB, p, grid, stream);
      return split == 2 ? launch_i8<4, false, 2>(tmA, tmB, p, grid, stream)
                        : launch_i8<4, false, 4>(tmA, tmB, p, grid, stream);
    }
    return GP_ERR_UNSUPPORTED;
  }
  if (p.w4) {
    switch (strip) {
      case 16: return launch_i8<2, true>(tmA, tmB, p, grid, stream);
      case 24: return launch_i8<3, true>(tmA, tmB, p, grid, stream);
      case 32: return launch_i8<4, true>(tmA, tmB, p, grid, stream);
      case 48: return launch_i8<6, true>(tmA, tmB, p, grid, stream);
      default: return launch_i8<8, true>(tmA, tmB, p, grid, stream);
    }
  }
  switch (strip) {
    case 16: return launch_i8<2, false>(tmA, tmB, p, grid, stream);
    case 24: return launch_i8<3, false>(tmA, tmB, p, grid, stream);
    case 32: return launch_i8<4, false>(tmA, tmB, p, grid, stream);
    case 48: return launch_i8<6, false>(tmA, tmB, p, grid, stream);
    default: return launch_i8<8, false>(tmA, tmB, p, grid, stream);
  }
}

}  // namespace gp
