// The offline preshuffle of B ("GEMM Optimization Guide", section 12: B is
// permuted once so that the GEMM's loads of B need no shuffle) and its
// inverse.
//
// Layout (this library's own; the guide's CDNA layout targets MFMA
// registers):
//   - B's bytes [N, Kb] are cut into R-row x 128-byte tiles: R = 128 for the
//     tcgen05 element types (BF16, E4M3, E2M1), R = 8 for INT8, whose
//     weight-streaming kernel gives each SM a strip of whole 8-row units.
//     Tile (tn, tk) is the R*128-byte block tn*(Kb/128) + tk, so the K tiles
//     of one band are contiguous.
//   - INT8 bytes are stored in offset binary (b XOR 0x80 = b + 128 as an
//     unsigned byte), the form the INT8 kernel hands to the MMA.  W4A8's
//     int4 B uses the same 8-row bands, with the nibbles of each 32-bit
//     word in offset binary and interleaved (w4_interleave).
//   - Row r of a tile lives at r*128.  Its 16-byte chunk c is stored at slot
//     c ^ (r % 8).  This is the 128-byte-swizzled K-major image that tcgen05
//     descriptors and TMA use, so one bulk copy lands a tile in shared memory
//     ready for the MMA, and 8 rows reading the same chunk hit 8 distinct
//     bank groups.  W4A8 stores chunk c at c ^ (r % 8) ^ 4 (r % 2) instead:
//     its kernel reads chunks c0 .. c0 + 3 of rows 2i and 2i + 1 in one
//     shared-memory phase, and the flip puts the two rows in different halves
//     of the banks (with c ^ (r % 8) alone every such read was 2-way
//     conflicted).
//   - E2M1 block scales ([N, K/32] bytes) follow the data region.  Per
//     (tn, tk) they take two 512-byte groups of four K blocks.  Inside a
//     group, (row r, block j) is at (r%32)*16 + (r/32)*4 + j%4: the 32-lane
//     x 16-byte image that tcgen05.cp copies into tensor memory.
#include "kernels.h"

namespace gp {

// rshift = log2(R).  w4: W4A8's slot rule, which also flips slot bit 2 on
// odd rows (see the header comment).
__device__ __forceinline__ int64_t packed_chunk_offset(int64_t n, int64_t cc, int64_t ktiles, int rshift, bool w4) {
  const int64_t tn = n >> rshift, r = n & ((int64_t(1) << rshift) - 1);
  const int64_t tk = cc >> 3, c = cc & 7;
  const int64_t mask = (r & 7) ^ (w4 ? (r & 1) << 2 : 0);
  return (((tn * ktiles + tk) << rshift) + r) * 128 + ((c ^ mask) << 4);
}

__device__ __forceinline__ int64_t packed_scale_offset(int64_t n, int64_t j, int64_t nblk) {
  const int64_t tiles_k = nblk >> 3;
  const int64_t tn = n >> 7, r = n & 127;
  const int64_t tk = j >> 3, jj = j & 7;
  const int64_t group = tn * (tiles_k * 2) + tk * 2 + (jj >> 2);
  return group * 512 + (r & 31) * 16 + (r >> 5) * 4 + (jj & 3);
}

// W4A8's int4 B: a 32-bit word of a row holds k0..k7 (two's complement
// nibbles at bits 4k).  Packed, each becomes u = b + 8 and k0..k7 move to
// bits 0, 16, 4, 20, 8, 24, 12, 28: (word >> 4j) & 0x000F000F is then the
// pair (k2j, k2j+1) as two fp16 bit patterns.
__device__ __forceinline__ uint32_t w4_interleave(uint32_t w) {
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out |= ((w >> (8 * j)) & 0xFu) << (4 * j);             // k = 2j
    out |= ((w >> (8 * j + 4)) & 0xFu) << (16 + 4 * j);    // k = 2j + 1
  }
  return out ^ 0x88888888u;
}

__device__ __forceinline__ uint32_t w4_deinterleave(uint32_t w) {
  w ^= 0x88888888u;
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out |= ((w >> (4 * j)) & 0xFu) << (8 * j);
    out |= ((w >> (16 + 4 * j)) & 0xFu) << (8 * j + 4);
  }
  return out;
}

// One warp per row of B; its lanes take consecutive 16-byte chunks, so a
// step reads 512 contiguous bytes of the row (pack) and writes whole
// 128-byte row segments of four tiles (the slot permutation stays inside a
// segment).  Each lane loads PACK_UNROLL chunks before it stores any, for
// more bytes in flight.  UNPACK runs the same walk in reverse.
constexpr int PACK_WARPS = 8, PACK_UNROLL = 4;

template <bool UNPACK>
__global__ void __launch_bounds__(32 * PACK_WARPS)
    pack_rows_kernel(const uint8_t* __restrict__ src, int64_t N, int64_t kbytes, int rshift, uint32_t bias, bool w4,
                     uint8_t* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int64_t cpr = kbytes >> 4;  // 16-byte chunks per row
  const int64_t ktiles = kbytes >> 7;
  for (int64_t n = (int64_t)blockIdx.x * PACK_WARPS + (threadIdx.x >> 5); n < N; n += (int64_t)gridDim.x * PACK_WARPS) {
    for (int64_t c0 = 0; c0 < cpr; c0 += 32 * PACK_UNROLL) {
      uint4 v[PACK_UNROLL];
#pragma unroll
      for (int u = 0; u < PACK_UNROLL; ++u) {
        const int64_t cc = c0 + u * 32 + lane;
        if (cc < cpr) {
          const int64_t off = UNPACK ? packed_chunk_offset(n, cc, ktiles, rshift, w4) : (n * cpr + cc) * 16;
          v[u] = *reinterpret_cast<const uint4*>(src + off);
        }
      }
#pragma unroll
      for (int u = 0; u < PACK_UNROLL; ++u) {
        const int64_t cc = c0 + u * 32 + lane;
        if (cc < cpr) {
          uint4 x = v[u];
          if (w4) {
            if (UNPACK)
              x.x = w4_deinterleave(x.x), x.y = w4_deinterleave(x.y), x.z = w4_deinterleave(x.z),
              x.w = w4_deinterleave(x.w);
            else
              x.x = w4_interleave(x.x), x.y = w4_interleave(x.y), x.z = w4_interleave(x.z), x.w = w4_interleave(x.w);
          } else {
            x.x ^= bias, x.y ^= bias, x.z ^= bias, x.w ^= bias;
          }
          const int64_t off = UNPACK ? (n * cpr + cc) * 16 : packed_chunk_offset(n, cc, ktiles, rshift, w4);
          *reinterpret_cast<uint4*>(dst + off) = x;
        }
      }
    }
  }
}

__global__ void pack_scale_kernel(const uint8_t* __restrict__ S, int64_t N, int64_t nblk, uint8_t* __restrict__ out) {
  const int64_t total = N * nblk;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / nblk, j = i - n * nblk;
    out[packed_scale_offset(n, j, nblk)] = S[i];
  }
}

__global__ void unpack_scale_kernel(const uint8_t* __restrict__ in, int64_t N, int64_t nblk, uint8_t* __restrict__ S) {
  const int64_t total = N * nblk;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / nblk, j = i - n * nblk;
    S[i] = in[packed_scale_offset(n, j, nblk)];
  }
}

static int grid_for(int64_t total, int threads) {
  int64_t g = (total + threads - 1) / threads;
  if (g > 65536) g = 65536;
  if (g < 1) g = 1;
  return (int)g;
}

int pack_b_launch(const uint8_t* B, const uint8_t* Bsf, int64_t N, int64_t kbytes, int64_t nblk, int layout,
                  uint8_t* out, cudaStream_t stream) {
  const int rshift = layout == PACK_TC ? 7 : 3;
  const uint32_t bias = layout == PACK_INT8 ? 0x80808080u : 0u;
  pack_rows_kernel<false><<<grid_for(N, PACK_WARPS), 32 * PACK_WARPS, 0, stream>>>(B, N, kbytes, rshift, bias,
                                                                                  layout == PACK_W4, out);
  if (Bsf != nullptr)
    pack_scale_kernel<<<grid_for(N * nblk, 256), 256, 0, stream>>>(Bsf, N, nblk, out + N * kbytes);
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

int unpack_b_launch(const uint8_t* packed, int64_t N, int64_t kbytes, int64_t nblk, int layout, uint8_t* B,
                    uint8_t* Bsf, cudaStream_t stream) {
  const int rshift = layout == PACK_TC ? 7 : 3;
  const uint32_t bias = layout == PACK_INT8 ? 0x80808080u : 0u;
  pack_rows_kernel<true><<<grid_for(N, PACK_WARPS), 32 * PACK_WARPS, 0, stream>>>(packed, N, kbytes, rshift, bias,
                                                                                 layout == PACK_W4, B);
  if (Bsf != nullptr)
    unpack_scale_kernel<<<grid_for(N * nblk, 256), 256, 0, stream>>>(packed + N * kbytes, N, nblk, Bsf);
  return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
}

}  // namespace gp
