// Internal interface between the C ABI layer (api.cu) and the kernels.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gemm_preshuffle.h"

namespace gp {

// Raises the dynamic shared-memory limit of `kern` (and, if given, its
// shared-memory carveout) on the current device the first time its launcher
// runs there.  `done` is that launcher's own per-device flag array (each
// launcher is a template instantiation for one kernel).  The flags are
// atomics because host threads may launch concurrently; two threads that both
// see a flag clear both set the attribute, which is harmless.
template <typename Kern>
inline int smem_attr_once(std::atomic<bool> (&done)[64], Kern kern, int bytes, int carveout = -1) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GP_ERR_CUDA;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return GP_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return GP_ERR_CUDA;
  if (carveout >= 0 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, carveout) != cudaSuccess)
    return GP_ERR_CUDA;
  if (dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return GP_OK;
}

struct TcParams {
  const uint8_t* Bp;      // packed B (data region)
  const uint8_t* Bsf;     // packed B scales (E2M1 only)
  const uint8_t* sfa;     // A scales, UE8M0 [M, K/32] row-major (E2M1 only)
  const float* sa;        // fp32 [M] row scales or null
  const float* sb;        // fp32 [N] column scales or null
  const float* bias;      // fp32 [N] epilogue bias or null (no epilogue)
  int act;                // epilogue activation after the bias (EpiAct)
  int out_f16;            // 1: C is IEEE fp16, 0: bf16
  uint32_t* status;       // device status word
  uint64_t wait_limit_ns; // bounded-wait limit
  int M, N, K;            // K in elements
  int ktiles;             // row bytes / 128
  int tiles_m, tiles_n, num_tiles;
  int debug_skip_load;    // 0 = off; i > 0: the producer skips its i-th stage load
  int b_constant;         // 1: B may be read before the previous kernel on the stream completes
  int raster_g;           // M tiles per group of the tile order (tile_coords)
};

struct I8Params {
  const uint8_t* Bp;      // packed B
  int32_t* C;             // [M, N] int32
  uint32_t* status;
  uint64_t wait_limit_ns;
  int M, N, K;
  int ktiles;             // K / 128
  int strip;              // rows of B per CTA (multiple of 16), the B box height
  int stages;
  int b_constant;         // 1: B may be read before the previous kernel on the stream completes
  int independent;        // 1: nothing in flight touches the operands; wait for the previous kernel only at exit
  int w4;                 // 1: B is int4 (W4A8), packed as PACK_W4
  int debug_skip_load;    // 0 = off; i > 0: the B producer stops before its i-th stage load
  int mg0;                // first group of 16 rows of A of this launch (grids hold <= 65535 groups)
  int split;              // CTAs of a cluster sharing one strip along K (1, 2, 4 or 8)
};

// Output tile t of a tiles_m x tiles_n grid, walked in groups of G M tiles
// (16 unless GP_RASTER_G sets it) so that concurrently running CTAs cover a
// compact block of C and share A rows and B columns in L2.
constexpr int kRasterG = 16;
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int G, int& mb, int& nb) {
  const int group_size = G * tiles_n;
  const int group = t / group_size;
  const int first_m = group * G;
  const int gm = min(tiles_m - first_m, G);
  const int r = t - group * group_size;
  mb = first_m + r % gm;
  nb = r / gm;
}

void tc_tile_choice(int64_t M, int64_t N, int num_sms, int* bm, int* bn);
// K tiles per ring stage of the tile kernel: 2 for 128 x 128 tiles (A then
// travels as one 3-D TMA box [2][128 rows][128 B] and B as one 32 KiB
// copy), 1 for the others (a 2-D A box).
int tc_kstep(int bm, int bn);
int tc_gemm_launch(int kind, int bm, int bn, const CUtensorMap& tmA, const CUtensorMap& tmC, TcParams p, int num_sms,
                   cudaStream_t stream);
// Pairs of CTAs (a 2-CTA cluster, tcgen05 cta_group::2) on 256 x BN tiles,
// BN = 128 or 256, in place of single-CTA 128 x 128 or 256 x 256 tiles.
// pair_choice returns the pair tile's BN, or 0 to keep the single-CTA tile.
// tmA views A as [K tiles][M rows][128 B] with a box of [kPairKstep][128 rows]
// [128 B]; tmB views packed B as [tiles][128 rows][128 B] with a box of
// [kPairKstep][BN/2 rows][128 B].
constexpr int kPairKstep = 2;
int pair_choice(int64_t M, int bm, int bn);
// Whether a 256 x 256 pair tile splits its K range over its two accumulator
// buffers (summed in fp32 by the epilogue) for a product of `ktiles` K tiles.
bool pair_ksplit(int ktiles);
// Few 256 x 256 tiles with a long K: a 4-CTA cluster per tile, two pairs
// (one per half of K) whose partials are summed through distributed shared
// memory.  The pair kernel's tensor maps with BN = 256, their K boxes of
// kXpairKstep tiles.
bool xpair_choice(int64_t M, int64_t N, int ktiles, int num_sms);
// Its tensor maps' boxes hold kXpairKstep K tiles (A: a 3-D box of 128 rows).
constexpr int kXpairKstep = 1;
int xpair_gemm_launch(int kind, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, TcParams p,
                      cudaStream_t stream);
int pair_gemm_launch(int kind, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                     TcParams p, int num_sms, cudaStream_t stream);
int splitk_choice(int64_t M, int64_t N, int64_t ktiles, int num_sms);
int splitk_gemm_launch(int kind, int split, const CUtensorMap& tmA, const CUtensorMap& tmC, TcParams p,
                       cudaStream_t stream);
// MXFP4: single-CTA 128 x 256 tiles, or (pair) 2-CTA clusters on 256 x 256
// tiles.  tmB and tmSFB are used by the pair form only: packed B as
// [tiles][128 rows][128 B] with a box of one tile, and B's packed scales as
// [bands][K steps][4][256 B] with a box of one K step of two bands.
bool mxf4_pair_choice(int64_t M);
int mxf4_gemm_launch(bool pair, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFB,
                     const CUtensorMap& tmC, TcParams p, int num_sms, cudaStream_t stream);
int i8_strip_rows(int N, int num_sms);
int i8_split_k(int64_t ctas, int ktiles, int strip, int num_sms);
int i8_gemm_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, I8Params p, int num_sms, cudaStream_t stream);

int quant_launch(const void* X, bool x_bf16, int64_t M, int64_t K, bool to_e2m1, void* Q, void* S, int num_sms,
                 uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

// Packed-B layouts: 128-row bands, bytes as given (tcgen05 types); 8-row
// bands in offset binary (INT8); 8-row bands, interleaved offset-binary
// nibbles (W4A8's int4 B).
enum PackLayout : int { PACK_TC = 0, PACK_INT8 = 1, PACK_W4 = 2 };
int pack_b_launch(const uint8_t* B, const uint8_t* Bsf, int64_t N, int64_t kbytes, int64_t nblk, int layout,
                  uint8_t* out, cudaStream_t stream);
int unpack_b_launch(const uint8_t* packed, int64_t N, int64_t kbytes, int64_t nblk, int layout, uint8_t* B,
                    uint8_t* Bsf, cudaStream_t stream);

}  // namespace gp
