// Split-K tcgen05 GEMM for products with few output tiles (for example
// 512 x 4096 x 4096 on 152 SMs).
//
// The "GEMM Optimization Guide", section 13, asks that the tiles fill the GPU
// ("tile_m x tile_n fills GPU (enough blocks)").  Here enough tiles would mean
// small tiles.  On GB300 each SM takes in operands at about 110 GB/s, so small
// tiles move too many bytes per flop.  Instead, every output tile is 256 x 256
// (two M=128 MMAs share each B stage) and its K range is split across a
// thread-block cluster of SPLIT CTAs.
//   - Main loop: the dense kernel's, over this CTA's K/SPLIT slice.  The
//     producer warp feeds a TMA / bulk ring, one thread issues the MMAs, and
//     a 512-column fp32 accumulator lives in TMEM.
//   - Reduce-scatter over distributed shared memory.  CTA r owns rows
//     [r*256/SPLIT, (r+1)*256/SPLIT) of the tile.  After its accumulator
//     completes, its ring is free; it tells every peer so (a remote mbarrier
//     arrive).  Once all peers are free, each epilogue warp works through
//     32-row x 32-column blocks of its TMEM rows that another CTA owns.  It
//     stages each 4 KiB block in its local buffer, with a row-XOR swizzle of
//     the 16-byte chunks, so the owner's reads are free of bank conflicts.
//     One cp.async.bulk shared::cta -> shared::cluster copy moves the block
//     into the owner's ring.  Remote stores from registers measured slower:
//     st.shared::cluster ~10x, st.async ~1.3x the whole product's time.
//   - Such a copy completes only on an mbarrier of the destination CTA; the
//     sender has no way to see when it has finished reading its staging
//     buffer.  So the owner acknowledges every block.  Each (sender, sending
//     warp, staging buffer) is one stream into the owner with its own
//     receive barrier (4 KiB per phase, 4 blocks per stream).  At the owner
//     one lane of the otherwise idle producer warp watches each stream: when
//     a block has landed it arms the next phase and arrives remotely on the
//     sender's `sent_free` barrier of that buffer, and after the stream's
//     last block it arrives on `recv_all`.  A sending warp reuses a staging
//     buffer only after the acknowledgement of the block it last held, and
//     waits for both buffers' last acknowledgements before it stages its own
//     output rows there.  Every lane watches one stream on its own, so no
//     owner waits on a stream behind another that is itself waiting.
//   - Owner epilogue: the owner adds its own partial and the SPLIT-1
//     received ones in a fixed order, so results are deterministic.  It
//     applies scale_a[m] * scale_b[n] (E4M3), rounds to bf16 and stores
//     through the swizzled staging buffer with TMA.
//
// Waits on mbarriers are bounded, as in the other kernels.  A cluster barrier
// right after barrier initialisation makes every peer's barriers valid before
// any remote arrive; every thread reaches it unconditionally.
#include <cstdlib>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

namespace {

constexpr int SK_THREADS = 192;
constexpr int SK_BM = 256, SK_BN = 256, SK_STAGES = 3;
constexpr int SK_A_BYTES = SK_BM * 128, SK_B_BYTES = SK_BN * 128;
constexpr int SK_STAGE_BYTES = SK_A_BYTES + SK_B_BYTES;
constexpr int SK_RING = SK_STAGES * SK_STAGE_BYTES;  // 192 KiB, reused as the receive buffer
constexpr int SK_EPI = 4 * 2 * 32 * 128;  // two 4 KiB staging buffers per epilogue warp
constexpr int SK_BAR = 512;               // mbarriers, the TMEM slot and the abort flag
constexpr int SK_BLOCKS_PER_STREAM = SK_BN / 32 / 2;  // 32-column blocks of a warp's rows per staging buffer
constexpr int SK_MAX_STREAMS = 16;
constexpr int SK_SMEM = SK_RING + SK_EPI + SK_BAR + 1024;
static_assert(SK_SMEM <= 232448, "shared memory budget");

}  // namespace

template <int KIND, int SPLIT>
__global__ void __launch_bounds__(SK_THREADS, 1)
    splitk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC, TcParams p) {
  constexpr int OWN = SK_BM / SPLIT;           // rows owned per CTA
  constexpr int SLOT_BYTES = OWN * SK_BN * 4;  // one peer's partial of the owned rows
  static_assert((SPLIT - 1) * SLOT_BYTES <= SK_RING, "receive buffer fits in the ring");
  // Streams into an owner: (peer slot, 32-row block of the owned rows, staging buffer).
  constexpr int NQ = OWN / 32;
  constexpr int NSTREAM = (SPLIT - 1) * NQ * 2;
  static_assert(NSTREAM <= SK_MAX_STREAMS && NSTREAM <= 32, "one watching lane per stream");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = base;
  uint8_t* s_b = s_a + SK_STAGES * SK_A_BYTES;
  uint8_t* s_recv = base;  // the ring, once the main loop is done
  uint8_t* s_epi = base + SK_RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_epi + SK_EPI);
  uint64_t* empty = full + SK_STAGES;
  uint64_t* accf = empty + SK_STAGES;
  uint64_t* ready = accf + 1;      // peers' rings are free (SPLIT-1 remote arrivals)
  uint64_t* drain = ready + 1;
  uint64_t* recv = drain + 1;      // [stream]: one incoming 4 KiB block per phase (tx bytes)
  uint64_t* recv_all = recv + SK_MAX_STREAMS;  // every stream's last block has landed
  uint64_t* sent_free = recv_all + 1;          // [epilogue warp][buffer]: the owner has the block
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sent_free + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = p.wait_limit_ns;
  const int rank = (int)cluster_ctarank();
  const int tile = blockIdx.x / SPLIT;
  const int mb = tile / p.tiles_n, nb = tile % p.tiles_n;
  const int ks = p.ktiles / SPLIT;  // K steps of this CTA
  const int k0 = rank * ks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SK_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(ready, SPLIT - 1);
    mbar_init(drain, 1);
    for (int i = 0; i < NSTREAM; ++i) mbar_init(&recv[i], 1);
    mbar_init(recv_all, NSTREAM);
    for (int i = 0; i < 8; ++i) mbar_init(&sent_free[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    // each stream's first block (its later phases are armed by the lane that
    // watches it, before the acknowledgement that lets the next block come)
    for (int i = 0; i < NSTREAM; ++i) mbar_arrive_expect_tx(&recv[i], 32 * 128);
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) tmem_alloc<512>(tmem_slot);
  if (threadIdx.x == 64) {
    for (int kt = k0; kt < k0 + ks && kt < k0 + SK_STAGES; ++kt) {
      prefetch_l2_tile_2d(&tmA, kt * 128, mb * SK_BM);
      for (int j = 0; j < SK_BN / 128; ++j)
        prefetch_l2_bulk(p.Bp + ((size_t)(nb * (SK_BN / 128) + j) * p.ktiles + kt) * 16384, 16384);
    }
  }
  // With constant weights the producer requests B for the first stages
  // before the wait on the previous kernel; A follows after.
  const int early = p.b_constant ? min(ks, SK_STAGES) : 0;
  if (threadIdx.x == 0) {  // the producer thread, which initialised the barriers
    for (int i = 0; i < early; ++i) {
      if (p.debug_skip_load == 1 + i) continue;  // fault injection: see the producer loop
      mbar_arrive_expect_tx(&full[i], SK_STAGE_BYTES);
      for (int j = 0; j < SK_BN / 128; ++j)
        bulk_load(s_b + i * SK_B_BYTES + j * 16384,
                  p.Bp + ((size_t)(nb * (SK_BN / 128) + j) * p.ktiles + k0 + i) * 16384, 16384, &full[i]);
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  cluster_sync_all();  // every peer's barriers are initialised before any remote arrive
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t issued = 0;
      bool ok = true;
      const uint8_t* bsrc = p.Bp + (size_t)nb * (SK_BN / 128) * p.ktiles * 16384;
      for (int i = 0; i < ks; ++i) {
        const int s = i % SK_STAGES;
        const uint32_t ph = (uint32_t)(i / SK_STAGES) & 1;
        const int kt = k0 + i;
        if (p.debug_skip_load == 1 + i) {
          // Fault injection (host-selected): this stage gets neither copies
          // nor the producer's arrival, so the waits on it must time out.
          ++issued;
          continue;
        }
        if (i < early) {  // a free stage whose B is already requested
          tma_load_2d(s_a + s * SK_A_BYTES, &tmA, kt * 128, mb * SK_BM, &full[s]);
          ++issued;
          continue;
        }
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, limit)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], SK_STAGE_BYTES);
        tma_load_2d(s_a + s * SK_A_BYTES, &tmA, kt * 128, mb * SK_BM, &full[s]);
        for (int j = 0; j < SK_BN / 128; ++j)
          bulk_load(s_b + s * SK_B_BYTES + j * 16384, bsrc + ((size_t)j * p.ktiles + kt) * 16384, 16384, &full[s]);
        ++issued;
      }
      if (!ok || *abort_flag) {
        const uint32_t n = issued < (uint32_t)SK_STAGES ? issued : (uint32_t)SK_STAGES;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t q = issued - 1 - i;
          if (p.debug_skip_load == 1 + (int)q) continue;  // nothing was issued for it
          volatile int never = 0;
          wait_bounded(&full[q % SK_STAGES], (q / SK_STAGES) & 1, &never, p.status, ST_TIMEOUT_DRAIN, limit);
        }
      }
    }
    __syncwarp();
    // ------------------------------------------------------------ acknowledgements
    // Lane i watches incoming stream i = (peer slot, 32-row block, buffer).
    if (lane < NSTREAM) {
      const int b = lane & 1;
      const int qi = (lane >> 1) % NQ;
      const int slot = (lane >> 1) / NQ;
      const int sender = slot < rank ? slot : slot + 1;
      const int quad = (rank * OWN + qi * 32) % 128 / 32;  // the sending warp's TMEM lane quarter
      const uint32_t ack = mapa_shared(smem_u32(&sent_free[quad * 2 + b]), (uint32_t)sender);
      bool ok = true;
      for (int j = 0; j < SK_BLOCKS_PER_STREAM && ok; ++j) {
        ok = wait_bounded(&recv[lane], (uint32_t)j & 1, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit);
        if (!ok) break;
        if (j + 1 < SK_BLOCKS_PER_STREAM) mbar_arrive_expect_tx(&recv[lane], 32 * 128);
        mbar_arrive_remote(ack);
      }
      if (ok) mbar_arrive(recv_all);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = (KIND == 0) ? 1u : 0u;  // bf16; fp16 (KIND 2) and e4m3 (KIND 1) are format 0
      constexpr uint32_t idesc = idesc_dense(fmt, fmt, 128, SK_BN);
      bool ok = true;
      for (int i = 0; i < ks; ++i) {
        const int s = i % SK_STAGES;
        const uint32_t ph = (uint32_t)(i / SK_STAGES) & 1;
        if (!wait_bounded(&full[s], ph, abort_flag, p.status, ST_TIMEOUT_MMA, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(s_a + s * SK_A_BYTES);
        const uint32_t b0 = smem_u32(s_b + s * SK_B_BYTES);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bdesc = smem_desc_sw128(b0 + 32 * k);
#pragma unroll
          for (int mh = 0; mh < 2; ++mh)
            umma<KIND>(tmem_base + (uint32_t)(mh * SK_BN), smem_desc_sw128(a0 + mh * 16384 + 32 * k), bdesc, idesc,
                       (i | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      if (ok) umma_commit(accf);
      umma_commit(drain);
      volatile int never = 0;
      wait_bounded(drain, 0, &never, p.status, ST_TIMEOUT_DRAIN, limit);
    }
  } else {
    // ------------------------------------------------------------ epilogue / reduce-scatter
    const int quad = warp & 3;
    bool ok = wait_bounded(accf, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit);
    tc_fence_after();
    // The main loop is over, so this CTA's ring is free: tell every peer.
    if (ok && warp == 2 && lane < SPLIT && lane != rank) mbar_arrive_remote(mapa_shared(smem_u32(ready), lane));
    if (ok) ok = wait_cluster_bounded(ready, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit);
    // Send every 32 x 32 block of TMEM rows held here that another CTA owns:
    // stage it locally (row `lane`, chunk q at slot q ^ (lane % 8)), then one
    // bulk copy into the owner's receive slot [c][row][32 fp32].
    uint8_t* stg = s_epi + (warp - 2) * 8192;
    const uint32_t stg_row = smem_u32(stg) + lane * 128;
    uint64_t* my_free = &sent_free[quad * 2];
    int nsent = 0;  // blocks sent by this warp; buffer nsent % 2 takes the next one
#pragma unroll 1
    for (int mh = 0; mh < 2 && ok; ++mh) {
      const int R0 = mh * 128 + quad * 32;  // first tile row of this warp's block in half mh
      const int owner = R0 / OWN;
      if (owner == rank) continue;
      const int slot = rank < owner ? rank : rank - 1;  // this CTA's slot at the owner
      const int lr0 = R0 - owner * OWN;
      const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(mh * SK_BN);
#pragma unroll 1
      for (int c = 0; c < SK_BN / 32 && ok; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tb + (uint32_t)(c * 32), r);
        tmem_ld_wait();
        const int b = nsent & 1;
        const uint32_t boff = (uint32_t)(b * 4096);
        // the owner has acknowledged the block this buffer held before
        if (nsent >= 2)
          ok = wait_cluster_bounded(&my_free[b], (uint32_t)((nsent >> 1) - 1) & 1, abort_flag, p.status,
                                    ST_TIMEOUT_EPILOGUE, limit);
        if (!ok) break;
        const int stream = (slot * NQ + lr0 / 32) * 2 + b;  // at the owner
        const uint32_t rbar = mapa_shared(smem_u32(&recv[stream]), (uint32_t)owner);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_v4(stg_row + boff + (uint32_t)((q ^ (lane & 7)) << 4), r[4 * q], r[4 * q + 1], r[4 * q + 2],
                       r[4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t dst = mapa_shared(
              smem_u32(s_recv + slot * SLOT_BYTES + c * (OWN * 128) + lr0 * 128), (uint32_t)owner);
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 4096, [%2];" ::"r"(
                  dst),
              "r"(smem_u32(stg) + boff), "r"(rbar)
              : "memory");
        }
        ++nsent;
      }
    }
    // Both staging buffers are reused below: wait for the acknowledgement of
    // the last block each of them held.
    for (int b = 0; b < 2 && ok; ++b) {
      const int uses = (nsent + 1 - b) / 2;  // blocks this warp sent from buffer b
      if (uses > 0)
        ok = wait_cluster_bounded(&my_free[b], (uint32_t)(uses - 1) & 1, abort_flag, p.status, ST_TIMEOUT_EPILOGUE,
                                  limit);
    }
    __syncwarp();
    // Owned rows: add the peers' partials, scale, round, store.
#pragma unroll 1
    for (int mh = 0; mh < 2; ++mh) {
      const int R0 = mh * 128 + quad * 32;  // first tile row of this warp in half mh
      if (R0 / OWN != rank) continue;
      if (ok) ok = wait_bounded(recv_all, 0, abort_flag, p.status, ST_TIMEOUT_EPILOGUE, limit);
      if (!ok) break;
      const int R = R0 + lane;
      const int lr = R - rank * OWN;
      const int row0 = mb * SK_BM + R0;
      const int m = row0 + lane;
      const float sa = (p.sa != nullptr && m < p.M) ? __ldg(p.sa + m) : 1.0f;
      const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(mh * SK_BN);
#pragma unroll 1
      for (int c = 0; c < SK_BN / 64; ++c) {
        const int n0 = nb * SK_BN + c * 64;
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tb + (uint32_t)(c * 64 + h * 32), r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
#pragma unroll
          for (int sl = 0; sl < SPLIT - 1; ++sl) {
            const uint8_t* rowp = s_recv + sl * SLOT_BYTES + (2 * c + h) * (OWN * 128) + lr * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 x = *reinterpret_cast<const float4*>(rowp + ((q ^ (lr & 7)) << 4));
              v[4 * q] += x.x;
              v[4 * q + 1] += x.y;
              v[4 * q + 2] += x.z;
              v[4 * q + 3] += x.w;
            }
          }
          uint32_t pk[16];
          epi_row32(v, sa, p.sb != nullptr ? p.sb + n0 + h * 32 : nullptr,
                    p.bias != nullptr ? p.bias + n0 + h * 32 : nullptr, p.act, p.out_f16 != 0, pk);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = h * 4 + q;
            st_shared_v4(stg_row + (uint32_t)(((chunk ^ (lane & 7)) * 16)), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
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
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging read; the writes complete with the grid
  }

  tc_fence_before();
  __syncthreads();
  // No CTA leaves while a peer may still write into its ring (after a
  // bounded wait gave up, copies may still be in flight); every thread gets
  // here, since all waits above are bounded.
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<512>(tmem_base);
  }
}

template <int KIND, int SPLIT>
static int launch_splitk(const CUtensorMap& tmA, const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
  auto kern = splitk_gemm_kernel<KIND, SPLIT>;
  static std::atomic<bool> attr_set[64];
  if (const int rc = smem_attr_once(attr_set, kern, SK_SMEM); rc != GP_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_tiles * SPLIT);
  cfg.blockDim = dim3(SK_THREADS);
  cfg.dynamicSmemBytes = SK_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmC, p) != cudaSuccess) return GP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int splitk_choice(int64_t M, int64_t N, int64_t ktiles, int num_sms) {
  // Split K over a cluster when 256 x 256 tiles alone would leave most SMs
  // idle and every CTA keeps at least 32 K steps: the reduce-scatter costs a
  // few microseconds per tile (measured ~5 us for 192 KiB per SM), so it
  // pays off only against a long main loop (at 16 steps per CTA the 128 x 128
  // tile path was faster: 21 us vs 23.5 us at 512 x 4096 x 4096 bf16).
  // GP_SPLITK=0 disables the path; GP_SPLITK=2 or 4 forces that split
  // where it is valid (for sweeps).
  static const int mode = [] {
    const char* e = std::getenv("GP_SPLITK");
    return e == nullptr ? -1 : std::atoi(e);
  }();
  if (mode == 0 || N % SK_BN != 0) return 1;
  const int64_t tiles = ((M + SK_BM - 1) / SK_BM) * (N / SK_BN);
  if (mode == 2 || mode == 4) {  // forced split (sweeps), where it is valid
    return (tiles * mode <= num_sms && ktiles % mode == 0 && ktiles / mode >= 4) ? mode : 1;
  }
  for (int split : {4, 2}) {
    if (tiles * split <= num_sms && tiles * split * 2 > num_sms && ktiles % split == 0 && ktiles / split >= 32)
      return split;
  }
  return 1;
}

int splitk_gemm_launch(int kind, int split, const CUtensorMap& tmA, const CUtensorMap& tmC, TcParams p,
                       cudaStream_t stream) {
  p.tiles_m = (p.M + SK_BM - 1) / SK_BM;
  p.tiles_n = p.N / SK_BN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  if (split == 4)
    return kind == 0 ? launch_splitk<0, 4>(tmA, tmC, p, stream)
           : kind == 1 ? launch_splitk<1, 4>(tmA, tmC, p, stream)
                       : launch_splitk<2, 4>(tmA, tmC, p, stream);
  if (split == 2)
    return kind == 0 ? launch_splitk<0, 2>(tmA, tmC, p, stream)
           : kind == 1 ? launch_splitk<1, 2>(tmA, tmC, p, stream)
                       : launch_splitk<2, 2>(tmA, tmC, p, stream);
  return GP_ERR_UNSUPPORTED;
}

}  // namespace gp
