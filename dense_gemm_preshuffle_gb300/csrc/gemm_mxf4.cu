// Block-scaled MXFP4 GEMM for sm_103a (tcgen05.mma kind::mxf4):
//
//   C[m,n] = sum_j 2^(ea[m,j]-127) 2^(eb[n,j]-127) sum_{k in block j} A[m,k] B[n,k]
//
// "GEMM Optimization Guide", section 8.2, counts MXFP4 operands as E2M1 with
// one 1-byte scale per 32 K elements of each operand.  The block scales are
// applied inside the tensor core: every MMA instruction consumes 64 K
// elements, i.e. two UE8M0 scales per row of A and of B (scale_vec::2X).
// The scales are read from tensor memory.
//
// The structure matches the dense tcgen05 kernel.  It is a persistent
// 128 x 256 tile loop with a TMA/bulk producer warp, a single-thread MMA
// warp and four epilogue warps.  It adds:
//   - Scale layout in shared memory and TMEM.  A K step (256 elements,
//     8 scale blocks) holds two 512-byte "atoms" of scales per 128 rows.  In
//     an atom, the scale of (row r, block j) sits at byte
//     (r%32)*16 + (r/32)*4 + j.  tcgen05.cp (32x128b, warpx4) copies an atom
//     into four TMEM columns, replicated in the four 32-lane quarters.  So
//     lane r%32 of quarter q holds rows r%32 + 32c in column c, and the MMA
//     reads column r/32 for row r.
//   - B's scales arrive already in that image.  gemm_preshuffle_b packs them
//     next to B, and the producer bulk-copies them with the B tile.
//   - A's scales are plain [M, K/32] bytes.  Warp 6 places them into the
//     atom layout with 4-byte cp.async copies, two stages ahead of the MMA.
//     After the copies land it fences them for the async proxy (tcgen05.cp
//     reads shared memory through it) and arrives on the stage's barrier.
//     A stage is therefore full after one producer arrival plus its
//     transaction bytes and one arrival from warp 6.
//   - The epilogue reads a tile's whole accumulator into registers (rounded
//     to packed bf16/fp16) before it stages and stores it, and frees the
//     accumulator in between, so the next tile's MMAs overlap the stores
//     (not with SiLU / GELU, whose cost before the release outweighs it).
//   - TMEM: one 256-column fp32 accumulator, plus one scale slot per ring
//     stage (A: 2 atoms x 4 columns; B: 2 atoms x 8 columns).  Warp 7
//     copies a stage's scales into its slot (tcgen05.cp) as soon as the
//     stage lands and commits them to the stage's "scales ready" barrier,
//     which the MMA thread waits on; its own MMAs are then not held behind
//     the copies.
//
// The pair form (PAIR = true) runs a 2-CTA cluster on a 256 x 256 tile with
// tcgen05 cta_group::2, as the dense pair kernel does.
//   - CTA r holds rows [256 mb + 128 r, +128) of A and the 128-row band
//     2 nb + r of B.  Each CTA so takes in 32 KiB of operands a K step for
//     the math of a 128 x 256 tile (48 KiB alone).
//   - Every copy of both CTAs completes on the even CTA's full barrier: TMA
//     loads of the cta_group::2 form, with B and its scales through tensor
//     maps.
//   - Both A-scale warps arrive on that barrier.  The odd CTA's arrival is a
//     relaxed remote arrive behind a release fence limited to its own
//     shared memory; a full cluster-scope release cost 2.3x.
//   - Each CTA holds the scales of all 256 columns of B and its own A-scale
//     rows.  A cta_group::2 tcgen05.cp, issued by the even CTA's scale-copy
//     warp, copies each CTA's shared memory into that CTA's TMEM.
//   - The even CTA's MMA thread issues M = 256 MMAs.  Its commits arrive on
//     the barriers of both CTAs.
//   - The epilogue warps free the accumulator the same way: a fence limited
//     to shared memory, then a relaxed remote arrive (5305 -> 5483 TFLOP/s).
//   - Eight epilogue warps (two per TMEM lane quarter, 128 columns each)
//     halve the time the single accumulator is held at each tile's end.
//   - Measured at 4096 x 8192 x 8192: 5708 TFLOP/s against 4911 for the
//     single-CTA 128 x 256 tiles on the same GPU.
#include <cstdlib>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

namespace {

constexpr int F4_BN = 256;
constexpr int F4_SF_LOOKAHEAD = 2;  // stages the A-scale warp keeps in flight

template <bool PAIR>
struct F4Cfg {
  // warps: producer, MMA, 4 epilogue warps (2-5), A-scale warp (6),
  // scale-copy warp (7); the pair form adds 4 epilogue warps (8-11)
  static constexpr int EPI_WARPS = PAIR ? 8 : 4;
  static constexpr int THREADS = 32 * (4 + EPI_WARPS);
  static constexpr int EPI_COLS = F4_BN / (EPI_WARPS / 4);  // accumulator columns per epilogue warp
  static constexpr int STAGES = PAIR ? 5 : 4;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = (PAIR ? F4_BN / 2 : F4_BN) * 128;  // this CTA's rows of B
  static constexpr int SFA_BYTES = 1024;          // 2 atoms
  static constexpr int SFB_BYTES = F4_BN * 8;      // (BN/128) bands x 2 atoms: all the tile's columns
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SFB_BYTES;  // one CTA's copies of a stage
  static constexpr int EPI_BYTES = EPI_WARPS * 32 * 128;
  static constexpr int ACC_COLS = F4_BN;
  static constexpr int SFA_COLS = 8;
  static constexpr int SFB_COLS = 2 * (F4_BN / 32);
  static constexpr int SF_COL0 = ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(ACC_COLS + STAGES * (SFA_COLS + SFB_COLS) <= TMEM_COLS, "tensor memory budget");
  static constexpr int BIAS_BYTES = EPI_WARPS * F4_BN * 4;  // each epilogue warp's copy of a tile's bias
  static constexpr int SMEM =
      STAGES * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) + EPI_BYTES + BIAS_BYTES + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ void f4_tile_coords(int t, int tiles_m, int tiles_n, int& mb, int& nb) {
  constexpr int G = 16;
  const int group_size = G * tiles_n;
  const int group = t / group_size;
  const int first_m = group * G;
  const int gm = min(tiles_m - first_m, G);
  const int r = t - group * group_size;
  mb = first_m + r % gm;
  nb = r / gm;
}

// Shared-memory descriptor of a 32-row x 16-byte block stored contiguously
// (no swizzle; 8-row core matrices 128 bytes apart), the source of tcgen05.cp.
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 16;   // leading byte offset
  d |= (uint64_t)(128u >> 4) << 32;   // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;             // fixed 0b001
  return d;                           // swizzle mode 0: none
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

}  // namespace

// tmB and tmSFB are used by the pair form only: packed B as [tiles][128 rows]
// [128 B] (box: one tile) and its packed scales as [bands][K steps][4][256 B]
// (box: one K step of two bands).
template <bool PAIR>
__global__ void __launch_bounds__(F4Cfg<PAIR>::THREADS, 1)
    mxf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmC, TcParams p) {
  using Cfg = F4Cfg<PAIR>;
  constexpr int F4_STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = base;
  uint8_t* s_b = s_a + F4_STAGES * Cfg::A_BYTES;
  uint8_t* s_sfa = s_b + F4_STAGES * Cfg::B_BYTES;
  uint8_t* s_sfb = s_sfa + F4_STAGES * Cfg::SFA_BYTES;
  uint8_t* s_epi = s_sfb + F4_STAGES * Cfg::SFB_BYTES;
  float* s_bias = reinterpret_cast<float*>(s_epi + Cfg::EPI_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_epi + Cfg::EPI_BYTES + Cfg::BIAS_BYTES);
  uint64_t* empty = full + F4_STAGES;
  uint64_t* accf = empty + F4_STAGES;
  uint64_t* acce = accf + 1;
  uint64_t* drain = acce + 1;
  uint64_t* sfr = drain + 1;             // [stage] scales of the stage are in TMEM
  uint64_t* sfdrain = sfr + F4_STAGES;   // the scale-copy warp's copies have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;
  const int nblk = p.K / 32;  // scale bytes per row of A
  // Pair form: this CTA's rank, the pair's tile sequence, the even CTA's
  // full barriers (every copy of both CTAs completes there).
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int cta0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // first tile
  const int ctas = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;    // tile stride
  const uint32_t full_leader = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;
  const int tile_rows = PAIR ? 256 : 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < F4_STAGES; ++s) {
      // producer (with tx bytes) + A-scale warp; the pair's even CTA also
      // counts the odd CTA's A-scale warp
      mbar_init(&full[s], PAIR ? 3 : 2);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, (PAIR ? 2 : 1) * Cfg::EPI_WARPS);
    mbar_init(drain, 1);
    for (int s = 0; s < F4_STAGES; ++s) mbar_init(&sfr[s], 1);
    mbar_init(sfdrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmC);
    if constexpr (PAIR) {
      prefetch_tensormap(&tmB);
      prefetch_tensormap(&tmSFB);
    }
  }
  if constexpr (PAIR) {
    if (warp == 1) tmem_alloc_pair<Cfg::TMEM_COLS>(tmem_slot);
  } else {
    if (warp == 1) tmem_alloc<Cfg::TMEM_COLS>(tmem_slot);
  }
  const size_t sf_band_bytes = (size_t)p.ktiles * 1024;  // packed B scales of one 128-row band
  // B data and scales of stage s of this CTA's tile (nb) at K step kt
  auto load_b = [&](int s, int nb, int kt) {
    if constexpr (PAIR) {
      const uint32_t bar = full_leader + (uint32_t)(s * 8);
      tma_load_3d_pair(s_b + s * Cfg::B_BYTES, &tmB, 0, 0, (2 * nb + (int)rank) * p.ktiles + kt, bar);
      tma_load_4d_pair(s_sfb + s * Cfg::SFB_BYTES, &tmSFB, 0, 0, kt, 2 * nb, bar);
      return;
    }
#pragma unroll
    for (int j = 0; j < F4_BN / 128; ++j) {
      const int band = nb * (F4_BN / 128) + j;
      bulk_load(s_b + s * Cfg::B_BYTES + j * 16384, p.Bp + ((size_t)band * p.ktiles + kt) * 16384, 16384, &full[s]);
      bulk_load(s_sfb + s * Cfg::SFB_BYTES + j * 1024, p.Bsf + (size_t)band * sf_band_bytes + (size_t)kt * 1024, 1024,
                &full[s]);
    }
  };
  // The even CTA's producer arms a stage with the bytes of both CTAs.
  constexpr uint32_t ARM_TX = (PAIR ? 2 : 1) * Cfg::STAGE_TX;
  auto load_a = [&](int s, int mb, int kt) {
    if constexpr (PAIR)
      tma_load_2d_pair(s_a + s * Cfg::A_BYTES, &tmA, kt * 128, mb * 256 + (int)rank * 128,
                       full_leader + (uint32_t)(s * 8));
    else
      tma_load_2d(s_a + s * Cfg::A_BYTES, &tmA, kt * 128, mb * 128, &full[s]);
  };
  bool bad = false;  // pair form: the two CTAs' TMEM allocations differ
  if constexpr (PAIR) {
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated before any remote access
    tc_fence_after();
    bad = *tmem_slot != ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), rank ^ 1u));
    if (bad && leader && threadIdx.x == 0) atomicOr(p.status, ST_BAD_LAUNCH);
  }
  // With constant weights the producer requests B (data and scales) for the
  // first stages of its first tile before the wait on the previous kernel.
  const int early = (!bad && p.b_constant && cta0 < p.num_tiles) ? min(p.ktiles, F4_STAGES) : 0;
  if (threadIdx.x == 0 && early > 0) {  // the producer thread, which initialised the barriers
    int mb, nb;
    f4_tile_coords(cta0, p.tiles_m, p.tiles_n, mb, nb);
    for (int kt = 0; kt < early; ++kt) {
      if (p.debug_skip_load == 1 + kt) continue;  // fault injection: see the producer loop
      if (leader) mbar_arrive_expect_tx(&full[kt], ARM_TX);
      load_b(kt, nb, kt);
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem_base = *tmem_slot;

  if (bad) {
    // nothing to do: fall through to the final barrier
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = cta0; t < p.num_tiles && ok; t += ctas) {
        int mb, nb;
        f4_tile_coords(t, p.tiles_m, p.tiles_n, mb, nb);
        for (int kt = 0; kt < p.ktiles; ++kt) {
          if (p.debug_skip_load == 1 + (int)issued) {
            // Fault injection (host-selected): this stage gets neither copies
            // nor the producer's arrival, so the waits on it must time out.
          } else if ((int)issued < early) {  // a free stage whose B is already requested
            load_a(s, mb, kt);
          } else {
            if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full[s], ARM_TX);
            load_a(s, mb, kt);
            load_b(s, nb, kt);
          }
          ++issued;
          if (++s == F4_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (leader && (!ok || *abort_flag)) {
        // Another role (or this one) gave up: wait (bounded) for the loads
        // still in flight, so nothing lands in shared memory after exit.  (The
        // pair's odd CTA cannot: its copies complete on the even CTA's
        // barriers, which this wait covers, or its other roles run into the
        // wait limit before the final barrier.)
        const uint32_t n = issued < (uint32_t)F4_STAGES ? issued : (uint32_t)F4_STAGES;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t q = issued - 1 - i;
          if (p.debug_skip_load == 1 + (int)q) continue;  // nothing was issued for it
          volatile int never = 0;
          wait_bounded(&full[q % F4_STAGES], (q / F4_STAGES) & 1, &never, p.status, ST_TIMEOUT_DRAIN, limit);
        }
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ A-scale warp
    // Lane l moves rows l + 32c (c = 0..3) of the tile: their 8 scale bytes
    // of this K step split into atom 0 (blocks 0-3) and atom 1 (blocks 4-7),
    // at byte l*16 + c*4 of each atom.
    uint32_t q = 0;       // stage sequence number (same order as the producer)
    uint32_t done = 0;    // stages already signalled
    bool ok = true;
    // Publish stage `st` on the even CTA's full barrier.  The copies have
    // landed and were made visible to the async proxy, which the even CTA's
    // tcgen05.cp reads them through.  In the pair, the release covers this
    // CTA's shared memory only.  A full release at cluster scope made the
    // MXFP4 product 2.3x slower.
    auto publish = [&](uint32_t st) {
      if constexpr (PAIR)
        mbar_arrive_remote_after_smem_writes(full_leader + st * 8);
      else
        mbar_arrive(&full[st]);
    };
    for (int t = cta0; t < p.num_tiles && ok; t += ctas) {
      int mb, nb;
      f4_tile_coords(t, p.tiles_m, p.tiles_n, mb, nb);
      for (int kt = 0; kt < p.ktiles; ++kt, ++q) {
        const int s = (int)(q % F4_STAGES);
        const uint32_t ph = (q / F4_STAGES) & 1;
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(s_sfa + s * Cfg::SFA_BYTES) + lane * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int m = mb * tile_rows + (int)rank * 128 + c * 32 + lane;
          const bool valid = m < p.M;
          const uint8_t* src = p.sfa + (size_t)(valid ? m : 0) * nblk + kt * 8;
          cp_async_4(dst + c * 4, src, valid ? 4u : 0u);
          cp_async_4(dst + 512 + c * 4, src + 4, valid ? 4u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (q + 1 >= (uint32_t)F4_SF_LOOKAHEAD) {
          // the stage issued LOOKAHEAD-1 steps ago has landed: publish it
          asm volatile("cp.async.wait_group %0;" ::"n"(F4_SF_LOOKAHEAD - 1) : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) publish(done % F4_STAGES);
          ++done;
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    __syncwarp();
    for (; done < q; ++done)
      if (lane == 0) publish(done % F4_STAGES);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int t = cta0; t < p.num_tiles && ok; t += ctas, ++local) {
        const bool freed = PAIR ? wait_cluster_bounded(acce, (uint32_t)(local & 1) ^ 1, abort_flag, p.status,
                                                       ST_TIMEOUT_MMA, limit)
                                : wait_bounded(acce, (uint32_t)(local & 1) ^ 1, abort_flag, p.status,
                                               ST_TIMEOUT_MMA, limit);
        if (!freed) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base;
        for (int kt = 0; kt < p.ktiles; ++kt) {
          if (!(PAIR ? wait_cluster_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)
                     : wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit))) {
            ok = false;
            break;
          }
          // the stage's scales are in TMEM (copied by warp 7)
          if (!wait_bounded(&sfr[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + Cfg::SF_COL0 + s * (Cfg::SFA_COLS + Cfg::SFB_COLS);
          const uint32_t sfb_t = sfa_t + Cfg::SFA_COLS;
          const uint32_t a0 = smem_u32(s_a + s * Cfg::A_BYTES);
          const uint32_t b0 = smem_u32(s_b + s * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t at = (uint32_t)(k >> 1);
            const uint32_t id = (uint32_t)(k & 1) * 2;
            if constexpr (PAIR)
              umma_mxf4_pair(d, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k),
                             idesc_mxf4(256, F4_BN, id, id), sfa_t + at * 4, sfb_t + at * (F4_BN / 32),
                             (kt | k) != 0 ? 1u : 0u);
            else
              umma_mxf4(d, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k), idesc_mxf4(128, F4_BN, id, id),
                        sfa_t + at * 4, sfb_t + at * (F4_BN / 32), (kt | k) != 0 ? 1u : 0u);
          }
          if constexpr (PAIR)
            umma_commit_pair(&empty[s], 0x3);
          else
            umma_commit(&empty[s]);
          if (++s == F4_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(accf, 0x3);
        else
          umma_commit(accf);
      }
      if constexpr (PAIR)
        umma_commit_pair(drain, 0x1);
      else
        umma_commit(drain);
      volatile int never = 0;
      wait_bounded(drain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ scale-copy warp
    // One lane copies each stage's scales from shared memory into that
    // stage's TMEM slot as soon as the stage lands, and commits the copies
    // to sfr[s].  The MMA thread then finds them in place: copies issued
    // from its own thread, right before the MMAs that read them, held the
    // tensor pipe (measured: 11% of the MXFP4 product).  A slot is free
    // again when its stage is refilled, since the producer refills a stage
    // only after the MMAs that read its slot have completed.
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = cta0; t < p.num_tiles && ok; t += ctas) {
        for (int kt = 0; kt < p.ktiles; ++kt) {
          if (!(PAIR ? wait_cluster_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)
                     : wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + Cfg::SF_COL0 + s * (Cfg::SFA_COLS + Cfg::SFB_COLS);
          const uint32_t sfb_t = sfa_t + Cfg::SFA_COLS;
          const uint32_t sfa_s = smem_u32(s_sfa + s * Cfg::SFA_BYTES);
          const uint32_t sfb_s = smem_u32(s_sfb + s * Cfg::SFB_BYTES);
#pragma unroll
          for (int at = 0; at < 2; ++at) {
            if constexpr (PAIR)
              tmem_cp_32x128b_warpx4_pair(sfa_t + at * 4, smem_desc_sf(sfa_s + at * 512));
            else
              tmem_cp_32x128b_warpx4(sfa_t + at * 4, smem_desc_sf(sfa_s + at * 512));
#pragma unroll
            for (int j = 0; j < F4_BN / 128; ++j) {
              if constexpr (PAIR)
                tmem_cp_32x128b_warpx4_pair(sfb_t + at * (F4_BN / 32) + j * 4,
                                            smem_desc_sf(sfb_s + j * 1024 + at * 512));
              else
                tmem_cp_32x128b_warpx4(sfb_t + at * (F4_BN / 32) + j * 4, smem_desc_sf(sfb_s + j * 1024 + at * 512));
            }
          }
          if constexpr (PAIR)
            umma_commit_pair(&sfr[s], 0x1);
          else
            umma_commit(&sfr[s]);
          if (++s == F4_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // every copy issued has completed before TMEM is released
      if constexpr (PAIR)
        umma_commit_pair(sfdrain, 0x1);
      else
        umma_commit(sfdrain);
      volatile int never = 0;
      wait_bounded(sfdrain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else if ((warp >= 2 && warp <= 5) || warp >= 8) {
    // ------------------------------------------------------------ epilogue
    // Epilogue warp e reads TMEM lane quarter warp % 4 and the accumulator
    // columns [col0, col0 + EPI_COLS): all 256 with four warps, one half
    // each with the pair form's eight, which halves the time the single
    // accumulator is held at each tile's end.
    constexpr int CPW = Cfg::EPI_COLS;
    const int e = warp < 8 ? warp - 2 : warp - 4;
    const int quad = warp & 3;
    const int col0 = (e / 4) * CPW;
    const bool early_release = p.act == EPI_ACT_NONE || p.act == EPI_ACT_RELU;
    uint8_t* stg = s_epi + e * 4096;
    const uint32_t stg_row = smem_u32(stg) + lane * 128;
    // The accumulator is free once both CTAs' epilogue warps have read it.
    // The reads have completed (tcgen05.wait::ld) and are fenced
    // (tcgen05.fence::before_thread_sync) before this arrive.  In the pair,
    // the release covers this CTA's shared memory only.  The single
    // accumulator holds back the next tile's MMAs, and a full cluster-scope
    // release cost 3% of the product.
    auto release = [&]() {
      if constexpr (PAIR)
        mbar_arrive_remote_after_smem_writes(mapa_shared(smem_u32(acce), 0));
      else
        mbar_arrive(acce);
    };
    int local = 0;
    for (int t = cta0; t < p.num_tiles; t += ctas, ++local) {
      int mb, nb;
      f4_tile_coords(t, p.tiles_m, p.tiles_n, mb, nb);
      // The tile's bias goes to this warp's shared-memory copy while the
      // tile's main loop runs (every thread would otherwise fetch all 256
      // values while the accumulator is held).  A copy per warp needs no
      // barrier across warps: the warp's own reads of the previous tile are
      // done (the __syncwarp below orders the overwrite after them).
      const float* bias_t = nullptr;
      if (p.bias != nullptr) {
        float4* sbuf = reinterpret_cast<float4*>(s_bias + e * F4_BN);
        const float4* src = reinterpret_cast<const float4*>(p.bias + nb * F4_BN);
        __syncwarp();
        sbuf[2 * lane] = __ldg(src + 2 * lane);
        sbuf[2 * lane + 1] = __ldg(src + 2 * lane + 1);
        __syncwarp();
        bias_t = reinterpret_cast<const float*>(sbuf);
      }
      if (!wait_bounded(accf, (uint32_t)(local & 1), abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit)) break;
      tc_fence_after();
      const int row0 = mb * tile_rows + (int)rank * 128 + quad * 32;
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16);
      if (early_release) {
        // The warp's whole share of the row (CPW outputs) is read from TMEM
        // and rounded into CPW/2 packed registers first, and the
        // accumulator is released: the next tile's MMAs then run while this
        // tile is staged and stored (the single accumulator otherwise holds
        // them back).
        uint32_t pk[CPW / 2];
#pragma unroll
        for (int c = 0; c < CPW / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)(col0 + c * 32), r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
          uint32_t q16[16];
          epi_row32<true>(v, 1.0f, nullptr, bias_t != nullptr ? bias_t + col0 + c * 32 : nullptr, p.act,
                          p.out_f16 != 0, q16);
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[c * 16 + e] = q16[e];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
#pragma unroll
        for (int c = 0; c < CPW / 64; ++c) {
          const int n0 = nb * F4_BN + col0 + c * 64;
          if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the staging tile
          __syncwarp();
#pragma unroll
          for (int chunk = 0; chunk < 8; ++chunk)
            st_shared_v4(stg_row + (uint32_t)(((chunk ^ (lane & 7)) * 16)), pk[c * 32 + 4 * chunk],
                         pk[c * 32 + 4 * chunk + 1], pk[c * 32 + 4 * chunk + 2], pk[c * 32 + 4 * chunk + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) {
            tma_store_2d(&tmC, n0, row0, stg);
            bulk_commit_group();
          }
        }
      } else {
        // SiLU / GELU: computing them for the whole row before the release
        // was slower than storing chunk by chunk and releasing at the end
#pragma unroll 1
        for (int c = 0; c < CPW / 64; ++c) {
          const int n0 = nb * F4_BN + col0 + c * 64;
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(col0 + c * 64 + h * 32), r);
            tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
            uint32_t q16[16];
            epi_row32<true>(v, 1.0f, nullptr, bias_t != nullptr ? bias_t + col0 + c * 64 + h * 32 : nullptr,
                            p.act, p.out_f16 != 0, q16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int chunk = h * 4 + q;
              st_shared_v4(stg_row + (uint32_t)(((chunk ^ (lane & 7)) * 16)), q16[4 * q], q16[4 * q + 1],
                           q16[4 * q + 2], q16[4 * q + 3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) {
            tma_store_2d(&tmC, n0, row0, stg);
            bulk_commit_group();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
      }
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes complete with the grid
  }

  tc_fence_before();
  if constexpr (PAIR) {
    __syncwarp();
    cluster_sync_all();  // no CTA touches its peer's shared or tensor memory after this
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair<Cfg::TMEM_COLS>(tmem_base);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
    }
  }
}

template <bool PAIR>
static int launch_mxf4(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFB,
                       const CUtensorMap& tmC, const TcParams& p, int grid, cudaStream_t stream) {
  using Cfg = F4Cfg<PAIR>;
  auto kern = mxf4_gemm_kernel<PAIR>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, Cfg::SMEM); rc != GP_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFB, tmC, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

bool mxf4_pair_choice(int64_t M) {
  // 256 x 256 pair tiles where a tile has rows for both CTAs (MXFP4
  // 4096 x 8192 x 8192: 5708 against 4911 TFLOP/s); GP_TC_PAIR=0 keeps the
  // single-CTA 128 x 256 tiles.
  static const bool enabled = [] {
    const char* e = std::getenv("GP_TC_PAIR");
    return !(e != nullptr && e[0] == '0');
  }();
  return enabled && M > 128;
}

int mxf4_gemm_launch(bool pair, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFB,
                     const CUtensorMap& tmC, TcParams p, int num_sms, cudaStream_t stream) {
  if (p.N % F4_BN != 0) return GP_ERR_SHAPE;
  p.tiles_m = (p.M + (pair ? 255 : 127)) / (pair ? 256 : 128);
  p.tiles_n = p.N / F4_BN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  if (pair) {
    const int pairs = num_sms / 2;
    return launch_mxf4<true>(tmA, tmB, tmSFB, tmC, p, 2 * (p.num_tiles < pairs ? p.num_tiles : pairs), stream);
  }
  return launch_mxf4<false>(tmA, tmB, tmSFB, tmC, p, p.num_tiles < num_sms ? p.num_tiles : num_sms, stream);
}

}  // namespace gp
