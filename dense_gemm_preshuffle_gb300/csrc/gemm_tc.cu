// tcgen05 GEMM for sm_103a: C[M,N] = A[M,K] . B[N,K]^T with B pre-packed.
//
// "GEMM Optimization Guide", sections 1-7, describes the method on AMD CDNA:
//   - tiles of C;
//   - a double-buffered K loop (section 2);
//   - a bank-conflict-free swizzle on both the write and read paths (section 3);
//   - B loaded straight from its preshuffled layout (sections 4.2 and 12);
//   - an epilogue that scales, casts and stores coalesced (section 7).
//
// This kernel is the Blackwell form of those steps.
//   - One persistent CTA per SM walks BM x BN output tiles in a grouped
//     order, so that concurrent CTAs share A rows and B columns in L2.
//   - Warp 0 is the producer.  Each ring stage holds KSTEP K steps.  Its
//     lane 1 issues one TMA load for the BM x 128-byte A tile of each (a 2-D
//     box, or one 3-D box of KSTEP K tiles; 128-byte swizzle, rows >= M and
//     K tiles past the end zero-filled).  Its lane 0 issues one plain bulk
//     copy per 128-row band of packed B, covering the stage's KSTEP
//     consecutive 16 KiB tiles, which already hold the swizzled image.  One
//     thread's copies complete one after another, so two issuers let A and
//     B travel in parallel; and each copy costs a fixed time whatever its
//     size, so 128 x 128 tiles take two K steps a stage (32 KiB copies,
//     7% faster at FP8 8192^3 than 16 KiB ones).  Data lands in an S-stage
//     shared-memory ring with full/empty mbarriers.
//   - Warp 1, one lane, issues tcgen05.mma.  Each 128-row half of the tile
//     has its own fp32 accumulator in tensor memory, and both halves
//     multiply the same B tile.
//   - The accumulators are double-buffered when they fit (2 x BM/128 x BN
//     <= 512 columns), so the epilogue of one tile overlaps the main loop of
//     the next.  tcgen05.commit releases each ring stage and signals a
//     finished accumulator.
//   - Warps 2-9 are the epilogue, two per 32-lane quarter of TMEM (a warp
//     may only read the quarter warp % 4), taking alternate 64-column
//     chunks.  Each reads its 32 TMEM lanes with tcgen05.ld and forms
//     acc * scale_a[m] * scale_b[n] (+ bias[n], then the activation of a
//     fused epilogue) in fp32.  It rounds to bf16 (RNE) and writes 32 x 64
//     staging tiles with the 128-byte swizzle: the 8 lanes of each store
//     phase hit 8 distinct bank groups (ncu: 0 store conflicts when no TMA
//     writes land beside the stores; extra wavefronts appear only where an
//     epilogue overlaps the next tile's ring copies).  A TMA store writes the tiles out and
//     clips rows >= M.  With the single 512-column accumulator of 256 x 256
//     tiles the epilogue is not overlapped, so eight warps halve it.
//
// Why BM = 256: on GB300 each SM takes in operands at about 110 GB/s from
// L2.  For the 128 x 256 tile that bound caps FP8 near 2.9 PFLOP/s.
// A 256 x 256 tile does twice the math per B byte: 64 KiB per K step
// instead of 2 x 48 KiB.  The cost is a single-buffered 512-column
// accumulator.
//
// KIND: 0 = bf16 x bf16 (kind::f16), 1 = e4m3 x e4m3 (kind::f8f6f4),
// 2 = fp16 x fp16 (kind::f16 with the f16 operand format).  One K
// step moves 128 bytes of each row (64 bf16 or 128 e4m3 elements), and one
// MMA instruction consumes 32 bytes of K.
#include <cstdlib>
#include <cstring>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

constexpr int TC_EPI_WARPS = 8;  // warps 2..9: two per TMEM lane quarter, alternate 64-column chunks
constexpr int TC_THREADS = 32 * (2 + TC_EPI_WARPS);

template <int BM, int BN, int STAGES, int KSTEP>
struct TcCfg {
  static constexpr int MH = BM / 128;  // 128-row halves (one MMA each)
  static constexpr int BANDS = BN / 128;  // 128-row bands of packed B
  static constexpr int A_BYTES = KSTEP * BM * 128;  // [K tile][BM rows][128 B]
  static constexpr int B_BYTES = KSTEP * BN * 128;  // [band][K tile][128 rows][128 B]
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = TC_EPI_WARPS * 32 * 128;  // one 32 x 64 bf16 staging tile per warp
  static constexpr int ACC_COLS = MH * BN;  // one accumulator buffer
  static constexpr int NBUF = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_NEED = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static_assert(TMEM_NEED <= 512, "tensor memory budget");
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int KIND, int BM, int BN, int STAGES, int KSTEP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC, TcParams p) {
  using Cfg = TcCfg<BM, BN, STAGES, KSTEP>;
  constexpr int NBUF = Cfg::NBUF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = base;
  uint8_t* s_b = s_a + STAGES * Cfg::A_BYTES;
  uint8_t* s_epi = s_b + STAGES * Cfg::B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_epi + Cfg::EPI_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;
  const int kstages = (p.ktiles + KSTEP - 1) / KSTEP;  // ring stages per tile (KSTEP K tiles each)
  // K tiles in stage ks (the last stage of a tile may hold fewer)
  auto stage_ktiles = [&](int ks) { return min(KSTEP, p.ktiles - ks * KSTEP); };
  // A of stage ks: one 2-D box (one K tile) or one 3-D box of KSTEP K tiles
  // (K tiles past the end read as zeros; the box is always complete)
  auto load_a = [&](int st, int mb, int ks) {
    if constexpr (KSTEP == 1)
      tma_load_2d(s_a + st * Cfg::A_BYTES, &tmA, ks * 128, mb * BM, &full[st]);
    else
      tma_load_3d(s_a + st * Cfg::A_BYTES, &tmA, 0, mb * BM, ks * KSTEP, &full[st]);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);  // the A and the B issuer
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], TC_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) tmem_alloc<Cfg::TMEM_COLS>(tmem_slot);
  if (threadIdx.x == 32 * 2 && (int)blockIdx.x < p.num_tiles) {
    // Warm L2 with the first K steps of this CTA's first tile while the
    // previous kernel may still run (a prefetch never changes later loads).
    int mb, nb;
    tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
    const int kpre = kstages < STAGES ? kstages : STAGES;
    for (int ks = 0; ks < kpre; ++ks) {
      if constexpr (KSTEP == 1)
        prefetch_l2_tile_2d(&tmA, ks * 128, mb * BM);
      else
        prefetch_l2_tile_3d(&tmA, 0, mb * BM, ks * KSTEP);
      for (int j = 0; j < Cfg::BANDS; ++j)
        prefetch_l2_bulk(p.Bp + ((size_t)(nb * Cfg::BANDS + j) * p.ktiles + ks * KSTEP) * 16384,
                         (uint32_t)stage_ktiles(ks) * 16384);
    }
  }
  // With constant weights the producer requests B for the first stages of
  // its first tile before the wait on the previous kernel; A follows after.
  const int early = (p.b_constant && (int)blockIdx.x < p.num_tiles) ? min(kstages, STAGES) : 0;
  if (threadIdx.x == 0 && early > 0) {  // the producer thread, which initialised the barriers
    int mb, nb;
    tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
    const uint8_t* bsrc = p.Bp + (size_t)nb * (BN / 128) * p.ktiles * 16384;
    const uint64_t pol_b = policy_evict_first();
    for (int ks = 0; ks < early; ++ks) {
      if (p.debug_skip_load == 1 + ks) continue;
      const uint32_t nk = (uint32_t)stage_ktiles(ks);
      mbar_arrive_expect_tx(&full[ks], Cfg::BANDS * nk * 16384);
      for (int j = 0; j < Cfg::BANDS; ++j)
        bulk_load_hint(s_b + ks * Cfg::B_BYTES + j * KSTEP * 16384, bsrc + ((size_t)j * p.ktiles + ks * KSTEP) * 16384,
                       nk * 16384, &full[ks], pol_b);
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // inputs may come from, and C may be read by, the previous kernel
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producers
    // Lane 0 issues the B copies and lane 1 the A copies: one thread's bulk
    // copies complete one after another, so the operands travel in parallel.
    if (lane < 2) {
      const bool is_b = lane == 0;
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      const uint64_t pol_b = policy_evict_first();  // B streams through once per M band
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
        const uint8_t* bsrc = p.Bp + (size_t)nb * Cfg::BANDS * p.ktiles * 16384;
        for (int ks = 0; ks < kstages; ++ks) {
          // B's first `early` stages are free and already requested
          const bool b_done = is_b && (int)issued < early;
          if (!b_done && !wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
            ok = false;
            break;
          }
          if (p.debug_skip_load == 1 + (int)issued) {
            // Fault injection (host-selected): leave this stage's barrier
            // without its arrivals, so the consumer's bounded wait times out.
          } else if (!is_b) {
            mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES);
            load_a(s, mb, ks);
          } else if (!b_done) {
            const uint32_t nk = (uint32_t)stage_ktiles(ks);
            mbar_arrive_expect_tx(&full[s], Cfg::BANDS * nk * 16384);
            for (int j = 0; j < Cfg::BANDS; ++j)
              bulk_load_hint(s_b + s * Cfg::B_BYTES + j * KSTEP * 16384,
                             bsrc + ((size_t)j * p.ktiles + ks * KSTEP) * 16384, nk * 16384, &full[s], pol_b);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok || *abort_flag) {
        // Another role (or this one) gave up: wait (bounded) for the loads
        // still in flight, so nothing lands in shared memory after exit.
        const uint32_t n = issued < (uint32_t)STAGES ? issued : (uint32_t)STAGES;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t q = issued - 1 - i;
          const int st = (int)(q % STAGES);
          const uint32_t par = (q / STAGES) & 1;
          volatile int never = 0;
          if (p.debug_skip_load == 1 + (int)q) continue;
          wait_bounded(&full[st], par, &never, p.status, ST_TIMEOUT_DRAIN, limit);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = (KIND == 0) ? 1u /*bf16*/ : 0u /*fp16 (kind::f16) or e4m3 (kind::f8f6f4)*/;
      // With one K tile per stage the bands of B sit back to back and one
      // MMA covers all BN columns; with KSTEP > 1 each band is its own
      // 128-column MMA.
      constexpr uint32_t idesc = idesc_dense(fmt, fmt, 128, KSTEP == 1 ? BN : 128);
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++local) {
        const int buf = local % NBUF;
        const uint32_t use = (uint32_t)(local / NBUF);
        if (!wait_bounded(&acce[buf], (use & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * Cfg::ACC_COLS);
        for (int ks = 0; ks < kstages; ++ks) {
          if (!wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(s_a + s * Cfg::A_BYTES);
          const uint32_t b0 = smem_u32(s_b + s * Cfg::B_BYTES);
          const int nk = stage_ktiles(ks);
          for (int kk = 0; kk < nk; ++kk) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = (ks | kk | k) != 0 ? 1u : 0u;
              if constexpr (KSTEP == 1) {
                const uint64_t bdesc = smem_desc_sw128(b0 + 32 * k);
#pragma unroll
                for (int mh = 0; mh < Cfg::MH; ++mh)
                  umma<KIND>(d + (uint32_t)(mh * BN), smem_desc_sw128(a0 + mh * 16384 + 32 * k), bdesc, idesc, acc);
              } else {
#pragma unroll
                for (int j = 0; j < Cfg::BANDS; ++j) {
                  const uint64_t bdesc = smem_desc_sw128(b0 + (j * KSTEP + kk) * 16384 + 32 * k);
#pragma unroll
                  for (int mh = 0; mh < Cfg::MH; ++mh)
                    umma<KIND>(d + (uint32_t)(mh * BN + j * 128),
                               smem_desc_sw128(a0 + kk * (BM * 128) + mh * 16384 + 32 * k), bdesc, idesc, acc);
                }
              }
            }
          }
          umma_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&accf[buf]);
      }
      // Make sure every issued MMA has completed before TMEM is released.
      umma_commit(drain);
      volatile int never = 0;
      wait_bounded(drain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access: quad*32 .. +31
    const int chalf = (warp - 2) / 4;  // this warp takes the 64-column chunks c with c % 2 == chalf
    uint8_t* stg = s_epi + (warp - 2) * 4096;
    const uint32_t stg_row = smem_u32(stg) + lane * 128;
    int local = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++local) {
      int mb, nb;
      tile_coords(t, p.tiles_m, p.tiles_n, p.raster_g, mb, nb);
      const int buf = local % NBUF;
      const uint32_t use = (uint32_t)(local / NBUF);
      if (!wait_bounded(&accf[buf], use & 1, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit)) break;
      tc_fence_after();
#pragma unroll 1
      for (int mh = 0; mh < Cfg::MH; ++mh) {
        const int row0 = mb * BM + mh * 128 + quad * 32;
        const int m = row0 + lane;
        const float sa = (p.sa != nullptr && m < p.M) ? __ldg(p.sa + m) : 1.0f;
        const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * Cfg::ACC_COLS + mh * BN);
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
              const int chunk = h * 4 + q;
              st_shared_v4(stg_row + (uint32_t)(((chunk ^ (lane & 7)) * 16)), pk[4 * q], pk[4 * q + 1],
                           pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) {
            tma_store_2d(&tmC, n0, row0, stg);
            bulk_commit_group();
          }
        }
      }
      // accumulator buffer is free once every lane's TMEM loads are done
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[buf]);
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes complete with the grid
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
  }
}

// ---------------------------------------------------------------- host side

template <int KIND, int BM, int BN, int STAGES, int KSTEP>
static int launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmC, const TcParams& p, int grid,
                     cudaStream_t stream) {
  using Cfg = TcCfg<BM, BN, STAGES, KSTEP>;
  auto kern = tc_gemm_kernel<KIND, BM, BN, STAGES, KSTEP>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, Cfg::SMEM); rc != GP_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmC, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

void tc_tile_choice(int64_t M, int64_t N, int num_sms, int* bm, int* bn) {
  // The tile shape with the least estimated time: waves (ceil(tiles / SMs))
  // x tile area / the shape's relative throughput, measured on GB300 with
  // full waves (FP8 8192^3): 256 x 256 1.0, 128 x 256 0.90, 128 x 128 0.66
  // (smaller tiles bring fewer flops per operand byte, and each SM takes in
  // operands at ~110 GB/s).  Ties go to the larger tile.  GP_TC_TILE
  // (256x256, 128x256 or 128x128) overrides, for sweeps, where N allows.
  static const int forced = [] {
    const char* e = std::getenv("GP_TC_TILE");
    if (e == nullptr) return 0;
    if (std::strcmp(e, "256x256") == 0) return 1;
    if (std::strcmp(e, "128x256") == 0) return 2;
    if (std::strcmp(e, "128x128") == 0) return 3;
    return 0;
  }();
  if (forced == 1 && N % 256 == 0) {
    *bm = 256, *bn = 256;
    return;
  }
  if (forced == 2 && N % 256 == 0) {
    *bm = 128, *bn = 256;
    return;
  }
  if (forced == 3) {
    *bm = 128, *bn = 128;
    return;
  }
  struct Shape {
    int bm, bn;
    double rate;
  };
  const Shape shapes[3] = {{256, 256, 1.0}, {128, 256, 0.90}, {128, 128, 0.66}};
  double best = 0.0;
  for (const Shape& t : shapes) {
    if (N % t.bn != 0) continue;
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * (N / t.bn);
    const int64_t waves = (tiles + num_sms - 1) / num_sms;
    const double cost = (double)waves * t.bm * t.bn / t.rate;
    if (best == 0.0 || cost < best * (1.0 - 1e-9)) {
      best = cost;
      *bm = t.bm, *bn = t.bn;
    }
  }
}

int tc_kstep(int bm, int bn) { return (bm == 128 && bn == 128) ? 2 : 1; }

int tc_gemm_launch(int kind, int bm, int bn, const CUtensorMap& tmA, const CUtensorMap& tmC, TcParams p, int num_sms,
                   cudaStream_t stream) {
  p.tiles_m = (p.M + bm - 1) / bm;
  p.tiles_n = p.N / bn;
  p.num_tiles = p.tiles_m * p.tiles_n;
  const int grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (bm == 256) {
    if (bn != 256) return GP_ERR_UNSUPPORTED;
    switch (kind) {
      case 0: return launch_tc<0, 256, 256, 3, 1>(tmA, tmC, p, grid, stream);
      case 1: return launch_tc<1, 256, 256, 3, 1>(tmA, tmC, p, grid, stream);
      default: return launch_tc<2, 256, 256, 3, 1>(tmA, tmC, p, grid, stream);
    }
  }
  switch (kind) {
    case 0:
      return bn == 256 ? launch_tc<0, 128, 256, 4, 1>(tmA, tmC, p, grid, stream)
                       : launch_tc<0, 128, 128, 3, 2>(tmA, tmC, p, grid, stream);
    case 1:
      return bn == 256 ? launch_tc<1, 128, 256, 4, 1>(tmA, tmC, p, grid, stream)
                       : launch_tc<1, 128, 128, 3, 2>(tmA, tmC, p, grid, stream);
    default:
      return bn == 256 ? launch_tc<2, 128, 256, 4, 1>(tmA, tmC, p, grid, stream)
                       : launch_tc<2, 128, 128, 3, 2>(tmA, tmC, p, grid, stream);
  }
}

}  // namespace gp
