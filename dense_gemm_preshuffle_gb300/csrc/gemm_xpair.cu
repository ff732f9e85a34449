// K split over two pairs of CTAs (one 4-CTA cluster per 256 x 256 tile) for
// C[M,N] = A[M,K] . B[N,K]^T with B pre-packed, for products with few
// output tiles and a long K (BF16 512 x 4096 x 4096: 32 tiles for 152 SMs).
//
// "GEMM Optimization Guide", section 13: the tiles must fill the GPU.  Small
// tiles would, but each SM takes in operands at only ~100-120 GB/s, and a
// 128 x 128 tile brings the fewest flops per byte.  A pair of CTAs on a
// 256 x 256 tile (tcgen05 cta_group::2, as in the pair kernel) brings twice
// as many: each CTA takes in 128 rows of A and 128 rows of B per K tile for
// the math of a 128 x 256 block.  This kernel gives each tile two such
// pairs, one per half of K, so 32 tiles occupy 128 SMs:
//   - Cluster rank r: sub = r & 1 is the CTA's half of the tile's rows (and
//     of B's bands, as in the pair kernel), half = r >> 1 its half of K.
//     Ranks {0, 1} and {2, 3} are the two pairs; each pair's even CTA
//     issues its MMAs and owns its ring barriers, exactly as in the pair
//     kernel, with every multicast mask shifted to the pair's ranks.
//   - Each pair accumulates its K half in a 128 x 256 fp32 block of each
//     CTA's tensor memory (256 columns).
//   - Exchange (reduce-scatter through distributed shared memory): CTA r and
//     its K peer r ^ 2 hold partials of the same 128 rows.  Half 0 stores
//     columns [0, 128) of the tile, half 1 columns [128, 256).  Once a CTA's
//     own MMAs are complete its ring is free; it tells the K peer so (one
//     remote arrival).  Each epilogue warp reads the peer's 64 columns of
//     its 32 rows from tensor memory, writes them to its own ring (8 KiB,
//     16-byte chunks XOR-swizzled by row so that the stores and the peer's
//     loads hit distinct banks), and one cp.async.bulk shared::cta ->
//     shared::cluster copy moves them into the peer's ring, completing on
//     the peer's `xrecv` barrier (64 KiB expected from the peer's 8 warps).
//     Every buffer is written once, so no acknowledgements are needed.
//   - Each epilogue warp then adds the received partial to its own 64
//     columns (fp32, round to nearest: a + b is the same in either order, so
//     the result does not depend on which half finishes first), applies the
//     scales / bias / activation, rounds, and stores through a swizzled
//     staging tile with TMA.
// Every wait is bounded.  A cluster barrier ends the kernel: after it every
// copy that will ever be issued has been issued, and when every partial has
// landed, no copy reads or writes a CTA's shared memory any more.  If any
// epilogue warp gave up on its peer's partial it marks all four CTAs before
// the barrier; then a CTA that gave up waits for the partial once more
// (bounded) and a second barrier follows.  The TMEM columns are then freed
// by both CTAs of each pair.
//
// KIND as in the tile kernel: 0 = bf16, 1 = e4m3, 2 = fp16.
#include <cstdlib>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

namespace {

constexpr int XP_EPI_WARPS = 8;  // warps 2..9: two per TMEM lane quarter, one 64-column chunk of each half
constexpr int XP_THREADS = 32 * (2 + XP_EPI_WARPS);
template <int KSTEP, int STAGES>
struct XpCfg {
  static constexpr int A_BYTES = KSTEP * 128 * 128;  // [K tile][128 rows][128 B]
  static constexpr int B_BYTES = KSTEP * 128 * 128;  // [K tile][128 rows of the tile's 256][128 B]
  static constexpr int RING = STAGES * (A_BYTES + B_BYTES);
};
// After the main loop the ring holds: the partial for the K peer (8 warps x
// 32 rows x 64 fp32), the peer's partial for this CTA, and the output
// staging (8 warps x 32 rows x 64 16-bit values).
constexpr int XP_SLOT = 32 * 64 * 4;
constexpr int XP_OUT_OFF = 0;
constexpr int XP_IN_OFF = XP_EPI_WARPS * XP_SLOT;
constexpr int XP_STG_OFF = 2 * XP_EPI_WARPS * XP_SLOT;
constexpr int XP_BAR_BYTES = 256;
constexpr uint32_t XP_TMEM_COLS = 256;

}  // namespace

template <int KIND, int KSTEP, int STAGES, int NP>
__global__ void __launch_bounds__(XP_THREADS, 1)
    xpair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, TcParams p) {
  using Cfg = XpCfg<KSTEP, STAGES>;
  constexpr int XP_STAGES = STAGES;
  constexpr int XP_A_BYTES = Cfg::A_BYTES;
  constexpr int XP_B_BYTES = Cfg::B_BYTES;
  constexpr int XP_RING = Cfg::RING;
  static_assert(XP_STG_OFF + XP_EPI_WARPS * 32 * 128 <= XP_RING, "exchange buffers fit in the ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = base;
  uint8_t* s_b = s_a + XP_STAGES * XP_A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + XP_RING);  // the pair's even CTA: both CTAs' copies
  uint64_t* empty = full + XP_STAGES;
  uint64_t* accf = empty + XP_STAGES;  // this pair's MMAs are complete
  uint64_t* xfree = accf + 1;          // the K peer's ring may receive this CTA's partial
  uint64_t* xrecv = xfree + 1;         // the K peer's partial has landed here
  uint64_t* drain = xrecv + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* fail = reinterpret_cast<volatile uint32_t*>(abort_flag + 1);  // set by any CTA of the cluster

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t sub = rank & 1u;    // rows [128 sub, +128) of the tile, band 2 nb + sub of B
  const uint32_t half = rank >> 1;   // K tiles [kt0, kt1)
  const uint32_t lead = rank & 2u;   // this pair's even CTA
  const uint32_t kpeer = rank ^ 2u;  // the same rows, the other half of K
  const bool leader = sub == 0;
  const uint16_t pair_mask = (uint16_t)(0x3u << lead);
  const uint64_t limit = p.wait_limit_ns;
  const int kt0 = (int)half * p.ktiles / 2;
  const int kt1 = ((int)half + 1) * p.ktiles / 2;
  const int kstages = (kt1 - kt0 + KSTEP - 1) / KSTEP;
  {
    // Launch self-check, uniform over the cluster: four CTAs a cluster, one
    // tile per cluster, a K tile for each half, and the ring in the dynamic
    // shared memory.  A mismatch returns the whole cluster before any
    // cluster-wide wait.
    uint32_t dyn, ncta;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
    const uint32_t need = (uint32_t)(reinterpret_cast<const volatile uint8_t*>(fail + 1) - smem_raw);
    if (ncta != 4 || (int)(blockIdx.x >> 2) >= p.num_tiles || p.ktiles < 2 || need > dyn ||
        (int)blockDim.x != XP_THREADS) {
      if (threadIdx.x == 0) atomicOr(p.status, ST_BAD_LAUNCH);
      pdl_wait();
      return;
    }
  }
  int mb, nb;
  tile_coords((int)(blockIdx.x >> 2), p.tiles_m, p.tiles_n, p.raster_g, mb, nb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < XP_STAGES; ++s) {
      mbar_init(&full[s], 2);  // the even CTA's A and B issuers (unused in the odd CTA)
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(xfree, 1);
    mbar_init(xrecv, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *fail = 0;
    fence_mbar_init();
    // the K peer's eight copies of 8 KiB complete this barrier's only phase
    mbar_arrive_expect_tx(xrecv, (uint32_t)(XP_EPI_WARPS * XP_SLOT));
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) tmem_alloc_pair<XP_TMEM_COLS>(tmem_slot);
  tc_fence_before();
  cluster_sync_all();  // every CTA's barriers initialised and TMEM allocated before any remote access
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t pair_base = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), rank ^ 1u));
  const bool bad = tmem_base != pair_base;
  if (bad && threadIdx.x == 0) atomicOr(p.status, ST_BAD_LAUNCH);

  const uint32_t full_lead = mapa_shared(smem_u32(full), lead);
  const int a_row = mb * 256 + (int)sub * 128;
  const int b_tile0 = (2 * nb + (int)sub) * p.ktiles;  // this band's first K tile in packed B
  auto load_a = [&](int st, int ks) {
    tma_load_3d_pair(s_a + st * XP_A_BYTES, &tmA, 0, a_row, kt0 + ks * KSTEP, full_lead + (uint32_t)(st * 8));
  };
  auto load_b = [&](int st, int ks) {
    tma_load_3d_pair(s_b + st * XP_B_BYTES, &tmB, 0, 0, b_tile0 + kt0 + ks * KSTEP,
                     full_lead + (uint32_t)(st * 8));
  };

  if (!bad && threadIdx.x == 32 * 2) {
    // warm L2 with the first stages while the previous kernel may still run
    const int kpre = kstages < XP_STAGES ? kstages : XP_STAGES;
    for (int ks = 0; ks < kpre; ++ks) {
      prefetch_l2_tile_3d(&tmA, 0, a_row, kt0 + ks * KSTEP);
      prefetch_l2_tile_3d(&tmB, 0, 0, b_tile0 + kt0 + ks * KSTEP);
    }
  }
  // With constant weights the B issuers request the first stages of B
  // before the wait on the previous kernel.
  // Two stages, not the whole ring: A's first copies, issued after the wait,
  // then queue behind fewer B copies (BF16 512 x 4096 x 4096: 18.37 against
  // 18.6 us with all six stages requested early, 18.5 with none).
  const int early = (!bad && p.b_constant) ? min(kstages, min(XP_STAGES, 2)) : 0;
  constexpr int np = NP;  // issuing lane pairs of the producer warp
  if (warp == 0 && lane < 2 * np && (lane & 1) == 0 && early > 0) {
    for (int ks = lane >> 1; ks < early; ks += np) {
      if (p.debug_skip_load == 1 + ks) continue;
      if (leader) mbar_arrive_expect_tx(&full[ks], 2 * XP_B_BYTES);
      load_b(ks, ks);
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // A may come from, and C may be read by, the previous kernel

  bool recv_ok = true;  // epilogue warps: the K peer's partial arrived
  if (bad) {
    // nothing to do: fall through to the cluster barriers
  } else if (warp == 0) {
    // ------------------------------------------------------------ producers
    // Lanes 2j and 2j + 1 issue this CTA's rows of B and of A for the stages
    // ks = j (mod NP): one thread's copies complete one after another, so
    // NP pairs of issuers keep more of the ring's copies moving.
    if (lane < 2 * np) {
      const bool is_b = (lane & 1) == 0;
      int ks = lane >> 1;
      bool ok = true;
      for (; ks < kstages; ks += np) {
        const int s = ks % XP_STAGES;
        const uint32_t ph = (uint32_t)(ks / XP_STAGES) & 1u;
        const bool b_done = is_b && ks < early;
        if (!b_done && !wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
          ok = false;
          break;
        }
        if (p.debug_skip_load == 1 + ks) {
          // Fault injection (host-selected): leave this stage's barrier
          // without its arrivals, so the waits on it time out.
        } else if (!is_b) {
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * XP_A_BYTES);
          load_a(s, ks);
        } else if (!b_done) {
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * XP_B_BYTES);
          load_b(s, ks);
        }
      }
      if (leader && (!ok || *abort_flag)) {
        // wait (bounded) for the loads still in flight, so nothing lands in
        // shared memory after exit
        for (int q = ks - np; q >= 0 && q >= ks - XP_STAGES; q -= np) {
          volatile int never = 0;
          if (p.debug_skip_load == 1 + q) continue;
          wait_bounded(&full[q % XP_STAGES], (uint32_t)(q / XP_STAGES) & 1u, &never, p.status, ST_TIMEOUT_DRAIN,
                       limit);
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t fmt = (KIND == 0) ? 1u /*bf16*/ : 0u /*fp16 (kind::f16) or e4m3 (kind::f8f6f4)*/;
      constexpr uint32_t idesc = idesc_dense(fmt, fmt, 256, 256);
      bool ok = true;
      for (int ks = 0; ks < kstages; ++ks) {
        const int s = ks % XP_STAGES;
        const uint32_t ph = (uint32_t)(ks / XP_STAGES) & 1u;
        if (!wait_cluster_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(s_a + s * XP_A_BYTES);
        const uint32_t b0 = smem_u32(s_b + s * XP_B_BYTES);
        // the last stage of a half may hold a K tile of the other half: not used
        const int nk = min(KSTEP, kt1 - (kt0 + ks * KSTEP));
        for (int kk = 0; kk < nk; ++kk) {  // K tile kk of the stage
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (ks | kk | k) != 0 ? 1u : 0u;
            umma_pair<KIND>(tmem_base, smem_desc_sw128(a0 + kk * 16384 + 32 * k),
                            smem_desc_sw128(b0 + kk * 16384 + 32 * k), idesc, acc);
          }
        }
        umma_commit_pair(&empty[s], pair_mask);
      }
      if (ok) umma_commit_pair(accf, pair_mask);
      // every issued MMA completes before either CTA of the pair frees TMEM
      umma_commit_pair(drain, (uint16_t)(1u << rank));
      volatile int never = 0;
      wait_bounded(drain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;        // TMEM lanes quad*32 .. +31: rows of this warp
    const int w8 = warp - 2;          // exchange slot
    const int chalf = w8 >> 2;        // chunk chalf of each half of the columns
    const int own_c = (int)half * 2 + chalf;        // 64-column chunk this CTA stores
    const int peer_c = (1 - (int)half) * 2 + chalf;  // chunk the K peer stores
    const uint32_t tlane = tmem_base + ((uint32_t)(quad * 32) << 16);
    const uint32_t row_off = (uint32_t)lane * 256;  // this lane's row in a [32][64 fp32] slot
    // (each wait's outcome is made uniform over the warp: the code under it
    // synchronises the warp)
    if (__all_sync(0xffffffffu, wait_bounded(accf, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit))) {
      tc_fence_after();
      // This CTA's ring is free (every MMA that read it, and so every copy
      // into it, is complete): the K peer may send its partial.
      if (w8 == 0 && lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(xfree), kpeer));
      // The K peer's columns of this warp's rows, to the outgoing slot.
      const uint32_t out = smem_u32(base + XP_OUT_OFF + w8 * XP_SLOT);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tlane + (uint32_t)(peer_c * 64 + h * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = h * 8 + q;  // 16-byte chunk of the 256-byte row
          st_shared_v4(out + row_off + (uint32_t)((j ^ (lane & 7)) * 16), r[4 * q], r[4 * q + 1], r[4 * q + 2],
                       r[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (wait_cluster_bounded(xfree, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit)) {
          const uint32_t dst = mapa_shared(smem_u32(base + XP_IN_OFF + w8 * XP_SLOT), kpeer);
          const uint32_t rbar = mapa_shared(smem_u32(xrecv), kpeer);
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  dst),
              "r"(out), "n"(XP_SLOT), "r"(rbar)
              : "memory");
        }
      }
      __syncwarp();
      // This CTA's own columns.
      float v[64];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tlane + (uint32_t)(own_c * 64 + h * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[h * 32 + e] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      // The K peer's partial of the same rows and columns (its warp w8 sent them).
      recv_ok = __all_sync(0xffffffffu, wait_bounded(xrecv, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit));
      if (recv_ok) {
        const uint32_t in = smem_u32(base + XP_IN_OFF + w8 * XP_SLOT) + row_off;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float4 x;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                       : "r"(in + (uint32_t)((j ^ (lane & 7)) * 16)));
          v[4 * j] += x.x;
          v[4 * j + 1] += x.y;
          v[4 * j + 2] += x.z;
          v[4 * j + 3] += x.w;
        }
        const int row0 = a_row + quad * 32;
        const int m = row0 + lane;
        const float sa = (p.sa != nullptr && m < p.M) ? __ldg(p.sa + m) : 1.0f;
        const int n0 = nb * 256 + own_c * 64;
        uint8_t* stg = base + XP_STG_OFF + w8 * (32 * 128);
        const uint32_t stg_row = smem_u32(stg) + (uint32_t)lane * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
          epi_row32(*reinterpret_cast<float(*)[32]>(&v[h * 32]), sa, p.sb != nullptr ? p.sb + n0 + h * 32 : nullptr,
                    p.bias != nullptr ? p.bias + n0 + h * 32 : nullptr, p.act, p.out_f16 != 0, pk);
          // 128-byte swizzle: 16-byte chunk c of row `lane` goes to slot c ^ (lane % 8)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c16 = h * 4 + q;
            st_shared_v4(stg_row + (uint32_t)((c16 ^ (lane & 7)) * 16), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                         pk[4 * q + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.M) {
          tma_store_2d(&tmC, n0, row0, stg);
          bulk_commit_group();
          bulk_wait_group_read<0>();  // the staging tile is read; the writes complete with the grid
        }
        __syncwarp();
      }
    } else {
      recv_ok = false;
    }
  }

  // A warp that gave up on its peer's partial marks all four CTAs, so that
  // after the barrier every CTA of the cluster takes the same path.
  if (!bad && warp >= 2 && !recv_ok && lane == 0)
    for (uint32_t r = 0; r < 4; ++r) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)fail), r), 1u);
  tc_fence_before();
  cluster_sync_all();  // every copy that will be issued has been issued
  // When every partial has landed, every copy between the CTAs is complete
  // (a copy's arrival on its destination's barrier follows its last read of
  // the source): no CTA's shared memory is touched by another after this.
  if (*fail != 0) {
    if (!bad && warp >= 2 && !recv_ok) {
      // this CTA gave up on its peer's partial: let any copy already issued
      // into its ring land before the peer or this CTA may exit
      volatile int never = 0;
      wait_bounded(xrecv, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
    cluster_sync_all();  // no copy touches any CTA's shared memory after this
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair<XP_TMEM_COLS>(tmem_base);
  }
}

// ---------------------------------------------------------------- host side

bool xpair_choice(int64_t M, int64_t N, int ktiles, int num_sms) {
  // A 4-CTA cluster per 256 x 256 tile (two pairs, one per half of K) when
  // that is one wave and each pair keeps at least 32 K tiles of 128 bytes:
  // the exchange (64 KiB in and out per CTA) then costs little against the
  // main loop.  GP_XPAIR=0 disables the path; GP_XPAIR=1 takes it wherever
  // it is valid (N a multiple of 256, M > 128, K of 2 tiles or more).
  static const int mode = [] {
    const char* e = std::getenv("GP_XPAIR");
    return (e == nullptr || *e == '\0') ? -1 : std::atoi(e);
  }();
  if (mode == 0 || N % 256 != 0 || M <= 128 || ktiles < 2) return false;
  if (mode == 1) return true;
  const int64_t tiles = ((M + 255) / 256) * (N / 256);
  return tiles * 4 <= num_sms && ktiles >= 64;
}

template <int KIND, int KSTEP, int STAGES, int NP>
static int launch_xpair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const TcParams& p,
                        cudaStream_t stream) {
  constexpr int XP_SMEM = XpCfg<KSTEP, STAGES>::RING + XP_BAR_BYTES + 1024;
  static_assert(XP_SMEM <= 232448, "shared memory budget");
  auto kern = xpair_gemm_kernel<KIND, KSTEP, STAGES, NP>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, XP_SMEM); rc != GP_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * p.num_tiles);
  cfg.blockDim = dim3(XP_THREADS);
  cfg.dynamicSmemBytes = XP_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int xpair_gemm_launch(int kind, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, TcParams p,
                      cudaStream_t stream) {
  p.tiles_m = (p.M + 255) / 256;
  p.tiles_n = p.N / 256;
  p.num_tiles = p.tiles_m * p.tiles_n;
  if ((int64_t)p.num_tiles * 4 > 0x7fffffff) return GP_ERR_SHAPE;
  // Six stages of one K tile (32 KiB a CTA): against three of two K tiles
  // 18.74 against 18.98 us at BF16 512 x 4096 x 4096, 28.68 against 29.06
  // at 512 x 4096 x 8192 (seven stages, 224 KiB: no better than three).
  static_assert(kXpairKstep == 1, "the ring below stages one K tile");
  // Two issuing lane pairs (even and odd stages): 18.45 against 18.65 us
  // at BF16 512 x 4096 x 4096 with one pair, 28.33 against 28.52 at
  // 512 x 4096 x 8192 (three pairs: in between).
  switch (kind) {
    case 0: return launch_xpair<0, 1, 6, 2>(tmA, tmB, tmC, p, stream);
    case 1: return launch_xpair<1, 1, 6, 2>(tmA, tmB, tmC, p, stream);
    default: return launch_xpair<2, 1, 6, 2>(tmA, tmB, tmC, p, stream);
  }
}

}  // namespace gp
