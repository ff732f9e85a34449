// Pairs of CTAs on one tile (tcgen05 cta_group::2) for C[M,N] = A[M,K] . B[N,K]^T
// with B pre-packed.
//
// "GEMM Optimization Guide", sections 1-7: tiles of C, a pipelined K loop fed
// from B's preshuffled layout, and a scale/cast epilogue.  This kernel runs
// those steps on the tensor cores of two SMs at once.  A single CTA's
// 256 x 256 tile fills all 512 TMEM columns with one fp32 accumulator, so its
// epilogue holds back the next tile's MMAs.  Two CTAs sharing a 256 x 256
// tile each hold 128 x 256, so they can keep two accumulator buffers and
// overlap each tile's epilogue with the next main loop.
//
// A 2-CTA cluster computes a 256 x BN tile, BN = 128 or 256:
//   - CTA r (its rank in the cluster) loads rows [256 mb + 128 r, +128) of A
//     and BN/2 rows of B: for BN = 128 rows [64 r, +64) of the tile's
//     128-row band of packed B (a contiguous 8 KiB half of each 16 KiB
//     packed tile, which keeps its 128-byte swizzle because 64 is a multiple
//     of 8), for BN = 256 the whole band 2 nb + r.  A CTA so takes in 24 KiB
//     a K tile for the math of a 128 x 128 tile (32 KiB alone), or 32 KiB
//     for that of a 128 x 256 tile (48 KiB alone).
//   - One thread of the even CTA issues tcgen05.mma.cta_group::2 with
//     M = 256, N = BN.  The MMA reads both CTAs' shared memory at the same
//     offsets and writes each CTA's 128 accumulator rows into that CTA's
//     tensor memory, at the same column address.
//   - Both CTAs' copies complete on the even CTA's `full` barrier (the
//     cta_group::2 form of the TMA load), whose two issuers expect the bytes
//     of both CTAs.  An odd-CTA thread that waited for its copies and then
//     signalled the even CTA took 8 us longer at 512 x 4096 x 4096 (28.9
//     against 20.5 us).
//   - The MMA thread's commits arrive on the barriers of both CTAs at once
//     (multicast): each ring stage's `empty` and each accumulator's `accf`.
//   - Both CTAs' epilogue warps arrive on the even CTA's `acce` barrier once
//     they have read an accumulator buffer.
//   - Tensor memory: the two CTAs' allocating warps together allocate
//     2 x BN columns in both SMs: two accumulator buffers, so the epilogue of
//     one tile overlaps the next main loop.  For BN = 256 that is all 512
//     columns, which a single CTA's 256 x 256 tile needs for one buffer.
//     The kernel checks that both CTAs received the same address; if not, it
//     does no work and reports GP_ERR_DEVICE_CHECK.
// Long K (KSPLIT = 2): each tile's K range is split in two halves, the first
// accumulated in one TMEM buffer and the second in the other, and the
// epilogue adds the halves in fp32 (round to nearest) before scaling.  The
// tensor core's own accumulation is coarser than a round-to-nearest fp32 sum:
// at FP8 8192^3 a single chain over all of K reached 8.8e-3 of the parity
// metric on outputs near zero, where an fp32 chain stays under 4e-3.  Two
// chains of half the length, with half the magnitude swing each, cut that
// error.  Each buffer then holds one half of every tile: the first half is
// signalled at mid-tile and the epilogue reads it into registers at once,
// freeing buffer 0 for the next tile's first half; buffer 1 is read, and
// freed, at the tile's end, half a tile before the next tile needs it.
// Every wait is bounded, as in the other kernels, and a cluster barrier before
// the end keeps each CTA's shared and tensor memory alive while its peer may
// still use them.  The odd CTA cannot wait for its own copies (they complete
// on the even CTA's barrier).  Each of its copies is either consumed by the
// MMA, or the even CTA gave up before consuming it; then the odd CTA's
// epilogue (waiting for that tile's accumulator) or its producer (waiting
// for a free stage) runs into the wait limit before the final barrier, far
// longer than any copy takes to land.
//
// KIND as in the single-CTA kernel: 0 = bf16, 1 = e4m3, 2 = fp16.
#include <cstdlib>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

namespace {

constexpr int PR_EPI_WARPS = 8;  // warps 2..9: two per TMEM lane quarter, alternate 64-column chunks
constexpr int PR_THREADS = 32 * (2 + PR_EPI_WARPS);

template <int BN, int KSTEP, int STAGES>
struct PairCfg {
  static constexpr int B_ROWS = BN / 2;                 // rows of B per CTA
  static constexpr int A_BYTES = KSTEP * 128 * 128;     // [K tile][128 rows][128 B]
  static constexpr int B_BYTES = KSTEP * B_ROWS * 128;  // [K tile][BN/2 rows][128 B]
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = PR_EPI_WARPS * 32 * 128;  // one 32 x 64 staging tile per epilogue warp
  static constexpr int ACC_COLS = BN;
  static constexpr uint32_t TMEM_COLS = 2 * BN;         // two accumulator buffers
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "tensor memory budget");
};

}  // namespace

template <int KIND, int BN, int KSTEP, int STAGES, int KSPLIT>
__global__ void __launch_bounds__(PR_THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, TcParams p) {
  using Cfg = PairCfg<BN, KSTEP, STAGES>;
  static_assert(KSPLIT == 1 || KSPLIT == 2, "one chain per buffer, or one tile's two halves");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = base;
  uint8_t* s_b = s_a + STAGES * Cfg::A_BYTES;
  uint8_t* s_epi = s_b + STAGES * Cfg::B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_epi + Cfg::EPI_BYTES);  // even CTA: both CTAs' copies
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint64_t* acce = accf + 2;           // even CTA only: both CTAs have read the buffer
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)(blockIdx.x >> 1);
  const int npairs = (int)(gridDim.x >> 1);
  const uint64_t limit = p.wait_limit_ns;
  const int kstages = (p.ktiles + KSTEP - 1) / KSTEP;
  auto stage_ktiles = [&](int ks) { return min(KSTEP, p.ktiles - ks * KSTEP); };
  // Copies complete on the even CTA's barrier; its two issuers expect both
  // CTAs' bytes.
  const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
  // This CTA's rows of A: one box of KSTEP K tiles (past the last K tile the
  // box reads zeros, so it is always complete).
  auto load_a = [&](int st, int mb, int ks) {
    tma_load_3d_pair(s_a + st * Cfg::A_BYTES, &tmA, 0, mb * 256 + (int)rank * 128, ks * KSTEP,
                     full_leader + (uint32_t)(st * 8));
  };
  // This CTA's BN/2 rows of B, with packed B viewed as [tiles][128 rows][128 B]:
  // KSTEP consecutive K tiles of one band.
  auto load_b = [&](int st, int nb, int ks) {
    const int y = BN == 128 ? (int)rank * 64 : 0;
    const int band = BN == 128 ? nb : 2 * nb + (int)rank;
    tma_load_3d_pair(s_b + st * Cfg::B_BYTES, &tmB, 0, y, band * p.ktiles + ks * KSTEP,
                     full_leader + (uint32_t)(st * 8));
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);  // the even CTA's A and B issuers (unused in the odd CTA)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 2 * PR_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) tmem_alloc_pair<Cfg::TMEM_COLS>(tmem_slot);
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated before any remote access
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t peer_base = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), rank ^ 1u));
  const bool bad = tmem_base != peer_base;
  if (bad && leader && threadIdx.x == 0) atomicOr(p.status, ST_BAD_LAUNCH);

  if (!bad && threadIdx.x == 32 * 2 && pair < p.num_tiles) {
    // Warm L2 with the first K steps of this CTA's first tile while the
    // previous kernel may still run (a prefetch never changes later loads).
    int mb, nb;
    tile_coords(pair, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
    const int kpre = kstages < STAGES ? kstages : STAGES;
    const int y = BN == 128 ? (int)rank * 64 : 0;
    const int band = BN == 128 ? nb : 2 * nb + (int)rank;
    for (int ks = 0; ks < kpre; ++ks) {
      prefetch_l2_tile_3d(&tmA, 0, mb * 256 + (int)rank * 128, ks * KSTEP);
      prefetch_l2_tile_3d(&tmB, 0, y, band * p.ktiles + ks * KSTEP);
    }
  }
  // With constant weights the B issuer requests B for the first stages of
  // its first tile before the wait on the previous kernel; A follows after.
  const int early = (!bad && p.b_constant && pair < p.num_tiles) ? min(kstages, STAGES) : 0;
  if (threadIdx.x == 0 && early > 0) {  // warp 0 lane 0, the B issuer
    int mb, nb;
    tile_coords(pair, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
    for (int ks = 0; ks < early; ++ks) {
      if (p.debug_skip_load == 1 + ks) continue;
      if (leader) mbar_arrive_expect_tx(&full[ks], 2 * Cfg::B_BYTES);
      load_b(ks, nb, ks);
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // inputs may come from, and C may be read by, the previous kernel

  if (bad) {
    // nothing to do: fall through to the final cluster barrier
  } else if (warp == 0) {
    // ------------------------------------------------------------ producers
    // Lane 0 issues this CTA's rows of B, lane 1 its rows of A.
    if (lane < 2) {
      const bool is_b = lane == 0;
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = pair; t < p.num_tiles && ok; t += npairs) {
        int mb, nb;
        tile_coords(t, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
        for (int ks = 0; ks < kstages; ++ks) {
          const bool b_done = is_b && (int)issued < early;
          if (!b_done && !wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
            ok = false;
            break;
          }
          if (p.debug_skip_load == 1 + (int)issued) {
            // Fault injection (host-selected): leave this stage's barrier
            // without its arrivals, so the waits on it time out.
          } else if (!is_b) {
            if (leader) mbar_arrive_expect_tx(&full[s], 2 * Cfg::A_BYTES);
            load_a(s, mb, ks);
          } else if (!b_done) {
            if (leader) mbar_arrive_expect_tx(&full[s], 2 * Cfg::B_BYTES);
            load_b(s, nb, ks);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (leader && (!ok || *abort_flag)) {
        // Wait (bounded) for the loads still in flight, so nothing lands in
        // shared memory after exit.
        const uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t q = issued - 1 - i;
          volatile int never = 0;
          if (p.debug_skip_load == 1 + (int)q) continue;
          wait_bounded(&full[q % STAGES], (q / STAGES) & 1, &never, p.status, ST_TIMEOUT_DRAIN, limit);
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t fmt = (KIND == 0) ? 1u /*bf16*/ : 0u /*fp16 (kind::f16) or e4m3 (kind::f8f6f4)*/;
      constexpr uint32_t idesc = idesc_dense(fmt, fmt, 256, BN);
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      // KSPLIT = 2: stages [0, kh) go to buffer 0 and [kh, kstages) to buffer 1
      const int kh = KSPLIT == 2 ? kstages / 2 : kstages;
      for (int t = pair; t < p.num_tiles && ok; t += npairs, ++local) {
        const int buf = KSPLIT == 2 ? 0 : local & 1;
        const uint32_t use = KSPLIT == 2 ? (uint32_t)local : (uint32_t)(local >> 1);
        if (!wait_cluster_bounded(&acce[buf], (use & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < kstages; ++ks) {
          if (KSPLIT == 2 && ks == kh) {
            // the first half is issued: signal it, then take buffer 1 once
            // the epilogue has read the previous tile's second half
            umma_commit_pair(&accf[0], 0x3);
            if (!wait_cluster_bounded(&acce[1], (use & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!wait_cluster_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool second = ks >= kh;  // KSPLIT = 2: the second half's chain
          const uint32_t d = tmem_base + (uint32_t)((second ? 1 : buf) * Cfg::ACC_COLS);
          const int k0 = second ? kh : 0;  // first stage of this chain
          const uint32_t a0 = smem_u32(s_a + s * Cfg::A_BYTES);
          const uint32_t b0 = smem_u32(s_b + s * Cfg::B_BYTES);
          const int nk = stage_ktiles(ks);
          for (int kk = 0; kk < nk; ++kk) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = ((ks - k0) | kk | k) != 0 ? 1u : 0u;
              umma_pair<KIND>(d, smem_desc_sw128(a0 + kk * 16384 + 32 * k),
                              smem_desc_sw128(b0 + kk * (Cfg::B_ROWS * 128) + 32 * k), idesc, acc);
            }
          }
          umma_commit_pair(&empty[s], 0x3);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair(&accf[KSPLIT == 2 ? 1 : buf], 0x3);
      }
      // Every issued MMA must complete before either CTA releases TMEM.
      umma_commit_pair(drain, 0x1);
      volatile int never = 0;
      wait_bounded(drain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;              // TMEM lanes this warp may access: quad*32 .. +31
    const int chalf = (warp - 2) / 4;       // this warp takes the 64-column chunks c with c % 2 == chalf
    uint8_t* stg = s_epi + (warp - 2) * 4096;
    const uint32_t stg_row = smem_u32(stg) + lane * 128;
    const uint32_t acce_leader = mapa_shared(smem_u32(acce), 0);
    int local = 0;
    for (int t = pair; t < p.num_tiles; t += npairs, ++local) {
      int mb, nb;
      tile_coords(t, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
      const int buf = KSPLIT == 2 ? 0 : local & 1;
      const uint32_t use = KSPLIT == 2 ? (uint32_t)local : (uint32_t)(local >> 1);
      if (!wait_bounded(&accf[buf], use & 1, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit)) break;
      tc_fence_after();
      const int row0 = mb * 256 + (int)rank * 128 + quad * 32;
      const int m = row0 + lane;
      const float sa = (p.sa != nullptr && m < p.M) ? __ldg(p.sa + m) : 1.0f;
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * Cfg::ACC_COLS);
      if constexpr (KSPLIT == 2) {
        // This warp's BN/2 columns (64-column chunks c = chalf, chalf + 2,
        // ...).  The first half's sums (buffer 0) are complete at mid-tile:
        // they are read into registers then and buffer 0 is freed, so the
        // next tile's first half never waits.  At the tile's end the second
        // half's sums (buffer 1) are added in fp32, 16 columns at a time,
        // rounded and staged; buffer 1 is freed after its last read, half a
        // tile before the next tile needs it.
        constexpr int NC = BN / 128;  // chunks of this warp
        float held[NC][64];
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          const int c = chalf + 2 * ci;
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(tbase + (uint32_t)(c * 64 + pc * 16), r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) held[ci][pc * 16 + e] = __uint_as_float(r[e]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_leader);  // buffer 0 read: the next tile may start
        if (!wait_bounded(&accf[1], use & 1, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit)) break;
        tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          const int c = chalf + 2 * ci;
          const int n0 = nb * BN + c * 64;
          if (lane == 0) bulk_wait_group_read<0>();  // the previous store from this staging tile has read it
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
              uint32_t r[16];
              tmem_ld_32x32b_x16(tbase + (uint32_t)(Cfg::ACC_COLS + c * 64 + h * 32 + pc * 16), r);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) held[ci][h * 32 + pc * 16 + e] += __uint_as_float(r[e]);
            }
            if (ci == NC - 1 && h == 1) {
              // this warp's last reads of buffer 1
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_remote(acce_leader + 8u);
            }
            uint32_t pk[16];
            epi_row32(*reinterpret_cast<float(*)[32]>(&held[ci][h * 32]), sa,
                      p.sb != nullptr ? p.sb + n0 + h * 32 : nullptr,
                      p.bias != nullptr ? p.bias + n0 + h * 32 : nullptr, p.act, p.out_f16 != 0, pk);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c16 = h * 4 + q;
              st_shared_v4(stg_row + (uint32_t)(((c16 ^ (lane & 7)) * 16)), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                           pk[4 * q + 3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) {
            tma_store_2d(&tmC, n0, row0, stg);
            bulk_commit_group();
          }
        }
        continue;
      }
#pragma unroll 1
      for (int c = chalf; c < BN / 64; c += 2) {
        const int n0 = nb * BN + c * 64;
        // the previous TMA store from this staging tile must have read it
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 64 + h * 32), r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
          uint32_t pk[16];
          epi_row32(v, sa, p.sb != nullptr ? p.sb + n0 + h * 32 : nullptr,
                    p.bias != nullptr ? p.bias + n0 + h * 32 : nullptr, p.act, p.out_f16 != 0, pk);
          // 128-byte swizzle: 16-byte chunk j of row `lane` goes to slot j ^ (lane % 8)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c16 = h * 4 + q;
            st_shared_v4(stg_row + (uint32_t)(((c16 ^ (lane & 7)) * 16)), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                         pk[4 * q + 3]);
          }
        }
        if (c + 2 >= BN / 64) {
          // this warp's last TMEM loads of the tile are done: free the buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acce_leader + (uint32_t)(buf * 8));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.M) {
          tma_store_2d(&tmC, n0, row0, stg);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes complete with the grid
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA touches its peer's shared or tensor memory after this
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair<Cfg::TMEM_COLS>(tmem_base);
  }
}

// ---------------------------------------------------------------- host side

template <int KIND, int BN, int KSTEP, int STAGES, int KSPLIT = 1>
static int launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const TcParams& p,
                       int grid, cudaStream_t stream) {
  using Cfg = PairCfg<BN, KSTEP, STAGES>;
  auto kern = pair_gemm_kernel<KIND, BN, KSTEP, STAGES, KSPLIT>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, Cfg::SMEM); rc != GP_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PR_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int pair_choice(int64_t M, int bm, int bn) {
  // Pairs replace the single-CTA 256 x 256 tiles when a tile has rows for
  // both CTAs: the pair double-buffers its accumulators, so each tile's
  // epilogue overlaps the next main loop (FP8 8192^3: 3165 -> 3319 TFLOP/s).
  // 256 x 128 pairs in place of 128 x 128 tiles measured the same as the
  // single-CTA kernel (BF16 512 x 4096 x 4096: 20.49 against 20.47 us), so
  // they are taken only with GP_TC_PAIR=1.  GP_TC_PAIR=0 disables pairs.
  static const int mode = [] {
    const char* e = std::getenv("GP_TC_PAIR");
    return (e == nullptr || *e == '\0') ? -1 : std::atoi(e);
  }();
  if (mode == 0 || M <= 128) return 0;
  if (bm == 256 && bn == 256) return 256;
  if (mode == 1 && bm == 128 && bn == 128) return 128;
  return 0;
}

bool pair_ksplit(int ktiles) {
  // Split each 256 x 256 tile's K range over the two accumulator buffers
  // from 64 K tiles of 128 bytes on (FP8 K >= 8192, 16-bit K >= 4096): the
  // tensor core's accumulation error grows with the chain's length.
  // GP_PAIR_KSPLIT=0 keeps one chain per tile, =1 splits every tile.
  static const int mode = [] {
    const char* e = std::getenv("GP_PAIR_KSPLIT");
    return (e == nullptr || *e == '\0') ? -1 : std::atoi(e);
  }();
  if (mode == 0) return false;
  return mode == 1 ? ktiles >= 2 * kPairKstep : ktiles >= 64;
}

int pair_gemm_launch(int kind, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                     TcParams p, int num_sms, cudaStream_t stream) {
  p.tiles_m = (p.M + 255) / 256;
  p.tiles_n = p.N / bn;
  p.num_tiles = p.tiles_m * p.tiles_n;
  const int pairs = num_sms / 2;
  const int grid = 2 * (p.num_tiles < pairs ? p.num_tiles : pairs);
  if (bn == 128) {
    switch (kind) {
      case 0: return launch_pair<0, 128, kPairKstep, 4>(tmA, tmB, tmC, p, grid, stream);
      case 1: return launch_pair<1, 128, kPairKstep, 4>(tmA, tmB, tmC, p, grid, stream);
      default: return launch_pair<2, 128, kPairKstep, 4>(tmA, tmB, tmC, p, grid, stream);
    }
  }
  if (bn == 256) {
    if (pair_ksplit(p.ktiles)) {
      switch (kind) {
        case 0: return launch_pair<0, 256, kPairKstep, 3, 2>(tmA, tmB, tmC, p, grid, stream);
        case 1: return launch_pair<1, 256, kPairKstep, 3, 2>(tmA, tmB, tmC, p, grid, stream);
        default: return launch_pair<2, 256, kPairKstep, 3, 2>(tmA, tmB, tmC, p, grid, stream);
      }
    }
    switch (kind) {
      case 0: return launch_pair<0, 256, kPairKstep, 3>(tmA, tmB, tmC, p, grid, stream);
      case 1: return launch_pair<1, 256, kPairKstep, 3>(tmA, tmB, tmC, p, grid, stream);
      default: return launch_pair<2, 256, kPairKstep, 3>(tmA, tmB, tmC, p, grid, stream);
    }
  }
  return GP_ERR_UNSUPPORTED;
}

}  // namespace gp
