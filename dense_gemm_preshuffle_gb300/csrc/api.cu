// C ABI of the preshuffle GEMM library (declared in include/gemm_preshuffle.h).
//
// This layer:
//   - validates every argument on the host before launching anything;
//   - builds the TMA tensor maps for A and C;
//   - picks the kernel (tcgen05 tile kernel, its 2-CTA pair form, split-K
//     over a cluster, block-scaled MXFP4 kernel, or the INT8
//     weight-streaming kernel) and launches it on the caller's stream.
//
// It owns no per-call memory.  Each device gets a 4-byte status word (a
// __device__ variable) and a cached SM count.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace gp {

__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int64_t l2_bytes = 0;
  uint32_t* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return GP_ERR_CUDA;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return GP_ERR_CUDA;
    d.l2_bytes = l2;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return GP_ERR_CUDA;
    d.status = static_cast<uint32_t*>(addr);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return GP_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return GP_OK;
}

int elem_bits(int dtype) {
  switch (dtype) {
    case GP_BF16: return 16;
    case GP_FP16: return 16;
    case GP_E4M3: return 8;
    case GP_INT8: return 8;
    case GP_E2M1: return 4;
    case GP_W4A8: return 4;  // the bits of B; A is int8
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int pack_layout(int dtype) { return dtype == GP_INT8 ? PACK_INT8 : dtype == GP_W4A8 ? PACK_W4 : PACK_TC; }

// Shape rules shared by the packer and the GEMM (N, K part).
int check_nk(int dtype, int64_t N, int64_t K, int64_t* kbytes) {
  const int bits = elem_bits(dtype);
  if (bits == 0) return GP_ERR_INVALID_ARG;
  if (N < 0 || K < 0 || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return GP_ERR_SHAPE;
  if ((K * bits) % 8 != 0) return GP_ERR_SHAPE;
  const int64_t kb = K * bits / 8;
  if (N % 128 != 0 || kb % 128 != 0) return GP_ERR_SHAPE;
  *kbytes = kb;
  return GP_OK;
}

int encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* ptr, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GP_OK : GP_ERR_CUDA;
}

uint64_t wait_limit_ns() {
  // Bounded-wait limit for the GEMM kernels; GP_WAIT_LIMIT_MS overrides the
  // 2 s default (tests shorten it to exercise the timeout path quickly).
  static std::atomic<uint64_t> cached{0};
  uint64_t v = cached.load();
  if (v == 0) {
    v = 2000000000ull;
    if (const char* e = std::getenv("GP_WAIT_LIMIT_MS")) {
      const long long ms = std::atoll(e);
      if (ms > 0) v = (uint64_t)ms * 1000000ull;
    }
    cached.store(v);
  }
  return v;
}

std::atomic<int> g_debug_skip_load{0};

// M tiles per group of the persistent tile order (tile_coords).  When the A
// rows of all the product's M tiles fit in a third of L2 beside the B bands
// being read, one group takes them all (each B band is then read once, its
// tiles one after another): FP8 5120 x 5120 x 8320 (20 M tiles, 42.6 MB of A)
// 132.3-132.9 us against 133.7 with groups of 16.  Otherwise groups of 16
// (kRasterG): at FP8 8192^3 all 32 M tiles (64 MiB of A) took 337.7 us
// against 321.7.  GP_RASTER_G overrides, for sweeps.
int raster_group(int64_t tiles_m, int64_t tile_rows, int64_t kbytes, int64_t l2_bytes) {
  static const int forced = [] {
    const char* e = std::getenv("GP_RASTER_G");
    const int v = e == nullptr ? 0 : std::atoi(e);
    return v > 0 ? v : 0;
  }();
  if (forced > 0) return forced;
  if (tiles_m > kRasterG && tiles_m * tile_rows * kbytes <= l2_bytes / 3) return (int)tiles_m;
  return kRasterG;
}

}  // namespace
}  // namespace gp

using namespace gp;

// C[m, n] = act(bias[n]) rounded to bf16 or fp16: the fused epilogue of an
// empty (K = 0) sum.
__global__ void epilogue_broadcast_kernel(const float* __restrict__ bias, int act, int64_t M, int64_t N, int out_f16,
                                          uint16_t* __restrict__ C) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = epi_act(bias[i % N], act);
    C[i] = out_f16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

extern "C" {

const char* gemm_status_string(int status) {
  switch (status) {
    case GP_OK: return "GP_OK";
    case GP_ERR_INVALID_ARG: return "GP_ERR_INVALID_ARG: null pointer or bad enum value";
    case GP_ERR_UNSUPPORTED: return "GP_ERR_UNSUPPORTED: dtype / scale mode / output combination not offered";
    case GP_ERR_SHAPE: return "GP_ERR_SHAPE: dimension rule violated";
    case GP_ERR_ALIGNMENT: return "GP_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case GP_ERR_CUDA: return "GP_ERR_CUDA: a CUDA call failed";
    case GP_ERR_DEVICE_TIMEOUT: return "GP_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel gave up";
    case GP_ERR_DEVICE_CHECK: return "GP_ERR_DEVICE_CHECK: a kernel's launch self-check failed; it computed nothing";
    default: return "unknown gp_status";
  }
}

int gemm_packed_b_bytes(int dtype, int64_t N, int64_t K, size_t* bytes_out) {
  if (bytes_out == nullptr) return GP_ERR_INVALID_ARG;
  int64_t kb = 0;
  const int rc = check_nk(dtype, N, K, &kb);
  if (rc != GP_OK) return rc;
  size_t total = (size_t)N * (size_t)kb;
  if (dtype == GP_E2M1) total += (size_t)N * (size_t)(K / 32);
  *bytes_out = total;
  return GP_OK;
}

int gemm_preshuffle_b(const void* B, const void* B_scales, int dtype, int64_t N, int64_t K, void* B_packed,
                      void* stream) {
  int64_t kb = 0;
  int rc = check_nk(dtype, N, K, &kb);
  if (rc != GP_OK) return rc;
  if (N == 0 || K == 0) return GP_OK;
  if (B == nullptr || B_packed == nullptr) return GP_ERR_INVALID_ARG;
  if ((dtype == GP_E2M1) != (B_scales != nullptr)) return GP_ERR_INVALID_ARG;
  if (!aligned16(B) || !aligned16(B_packed)) return GP_ERR_ALIGNMENT;
  DeviceInfo* d = nullptr;
  if ((rc = device_info(&d)) != GP_OK) return rc;
  return pack_b_launch(static_cast<const uint8_t*>(B), static_cast<const uint8_t*>(B_scales), N, kb, K / 32,
                       pack_layout(dtype), static_cast<uint8_t*>(B_packed), static_cast<cudaStream_t>(stream));
}

int gemm_unpack_b(const void* B_packed, int dtype, int64_t N, int64_t K, void* B_out, void* B_scales_out,
                  void* stream) {
  int64_t kb = 0;
  int rc = check_nk(dtype, N, K, &kb);
  if (rc != GP_OK) return rc;
  if (N == 0 || K == 0) return GP_OK;
  if (B_packed == nullptr || B_out == nullptr) return GP_ERR_INVALID_ARG;
  if (dtype == GP_E2M1 && B_scales_out == nullptr) return GP_ERR_INVALID_ARG;
  if (!aligned16(B_out) || !aligned16(B_packed)) return GP_ERR_ALIGNMENT;
  DeviceInfo* d = nullptr;
  if ((rc = device_info(&d)) != GP_OK) return rc;
  return unpack_b_launch(static_cast<const uint8_t*>(B_packed), N, kb, K / 32, pack_layout(dtype),
                         static_cast<uint8_t*>(B_out),
                         dtype == GP_E2M1 ? static_cast<uint8_t*>(B_scales_out) : nullptr,
                         static_cast<cudaStream_t>(stream));
}

int gemm_run(const void* A, const void* B_packed, int dtype, int64_t M, int64_t N, int64_t K, int scale_mode,
             const void* scale_a, const void* scale_b, void* C, int c_dtype, void* stream) {
  return gemm_run_ex(A, B_packed, dtype, M, N, K, scale_mode, scale_a, scale_b, GP_EPI_NONE, nullptr, C, c_dtype,
                     GP_RUN_DEFAULT, stream);
}

int gemm_run_ex(const void* A, const void* B_packed, int dtype, int64_t M, int64_t N, int64_t K, int scale_mode,
                const void* scale_a, const void* scale_b, int epilogue, const void* bias, void* C, int c_dtype,
                unsigned flags, void* stream) {
  if ((flags & ~(unsigned)(GP_RUN_B_CONSTANT | GP_RUN_INDEPENDENT)) != 0) return GP_ERR_INVALID_ARG;
  const int independent = (flags & GP_RUN_INDEPENDENT) ? 1 : 0;
  const int b_constant = (flags & GP_RUN_B_CONSTANT) || independent ? 1 : 0;
  if (epilogue < GP_EPI_NONE || epilogue > GP_EPI_BIAS_GELU) return GP_ERR_INVALID_ARG;
  if ((epilogue == GP_EPI_NONE) != (bias == nullptr)) return GP_ERR_INVALID_ARG;
  const bool float_out = c_dtype == GP_BF16 || c_dtype == GP_FP16;
  if (epilogue != GP_EPI_NONE && !float_out) return GP_ERR_UNSUPPORTED;  // float outputs only
  // ---- combination
  const bool combo_ok = (dtype == GP_BF16 && scale_mode == GP_SCALE_NONE && float_out) ||
                        (dtype == GP_FP16 && scale_mode == GP_SCALE_NONE && float_out) ||
                        (dtype == GP_E4M3 && scale_mode == GP_SCALE_ROWCOL_F32 && float_out) ||
                        (dtype == GP_E4M3 && scale_mode == GP_SCALE_NONE && float_out) ||
                        (dtype == GP_E2M1 && scale_mode == GP_SCALE_BLOCK32_UE8M0 && float_out) ||
                        (dtype == GP_INT8 && scale_mode == GP_SCALE_NONE && c_dtype == GP_INT32) ||
                        (dtype == GP_W4A8 && scale_mode == GP_SCALE_NONE && c_dtype == GP_INT32);
  if (elem_bits(dtype) == 0 || scale_mode < GP_SCALE_NONE || scale_mode > GP_SCALE_BLOCK32_UE8M0 ||
      (!float_out && c_dtype != GP_INT32))
    return GP_ERR_INVALID_ARG;
  if (!combo_ok) return GP_ERR_UNSUPPORTED;
  // ---- shapes
  int64_t kb = 0;
  int rc = check_nk(dtype, N, K, &kb);
  if (rc != GP_OK) return rc;
  if (M < 0 || M >= (int64_t(1) << 31)) return GP_ERR_SHAPE;
  // the exact result must fit int32 for every input: K * 128 * 128 < 2^31
  // (int8 x int8) and K * 128 * 8 < 2^31 (int8 x int4)
  if (dtype == GP_INT8 && K >= 131072) return GP_ERR_SHAPE;
  if (dtype == GP_W4A8 && K >= 2097152) return GP_ERR_SHAPE;
  const size_t c_elem = c_dtype == GP_INT32 ? 4 : 2;
  if (M == 0 || N == 0) return GP_OK;  // empty output
  // ---- pointers
  if (C == nullptr) return GP_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B_packed == nullptr)) return GP_ERR_INVALID_ARG;
  if (scale_mode == GP_SCALE_ROWCOL_F32 && (scale_a == nullptr || scale_b == nullptr)) return GP_ERR_INVALID_ARG;
  if (scale_mode == GP_SCALE_BLOCK32_UE8M0 && (scale_a == nullptr || scale_b != nullptr)) return GP_ERR_INVALID_ARG;
  if (scale_mode == GP_SCALE_NONE && (scale_a != nullptr || scale_b != nullptr)) return GP_ERR_INVALID_ARG;
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B_packed)))) return GP_ERR_ALIGNMENT;
  if (scale_mode == GP_SCALE_ROWCOL_F32 && (!aligned16(scale_a) || !aligned16(scale_b))) return GP_ERR_ALIGNMENT;
  if (scale_mode == GP_SCALE_BLOCK32_UE8M0 && !aligned16(scale_a)) return GP_ERR_ALIGNMENT;
  if (bias != nullptr && !aligned16(bias)) return GP_ERR_ALIGNMENT;

  DeviceInfo* d = nullptr;
  if ((rc = device_info(&d)) != GP_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // empty sum: C = 0, or act(bias[n]) on every row with an epilogue
    if (epilogue == GP_EPI_NONE)
      return cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * c_elem, st) == cudaSuccess ? GP_OK : GP_ERR_CUDA;
    const int act = epilogue == GP_EPI_BIAS_RELU ? EPI_ACT_RELU
                    : epilogue == GP_EPI_BIAS_SILU ? EPI_ACT_SILU
                    : epilogue == GP_EPI_BIAS_GELU ? EPI_ACT_GELU
                                                   : EPI_ACT_NONE;
    const int64_t total = M * N;
    const int blocks = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
    epilogue_broadcast_kernel<<<blocks, 256, 0, st>>>(static_cast<const float*>(bias), act, M, N,
                                                      c_dtype == GP_FP16 ? 1 : 0, static_cast<uint16_t*>(C));
    return cudaGetLastError() == cudaSuccess ? GP_OK : GP_ERR_CUDA;
  }

  if (dtype == GP_INT8 || dtype == GP_W4A8) {
    const bool w4 = dtype == GP_W4A8;
    I8Params p{};
    p.Bp = static_cast<const uint8_t*>(B_packed);
    p.C = static_cast<int32_t*>(C);
    p.status = d->status;
    p.wait_limit_ns = wait_limit_ns();
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.ktiles = (int)(K / 128);  // 128-element K tiles of A (int8: K bytes a row)
    p.strip = i8_strip_rows((int)N, d->num_sms);
    p.split = i8_split_k(((N + p.strip - 1) / p.strip) * ((M + 15) / 16), p.ktiles, p.strip, d->num_sms);
    p.b_constant = b_constant;
    p.independent = independent;
    p.w4 = w4 ? 1 : 0;
    p.debug_skip_load = g_debug_skip_load.exchange(0);
    const int64_t b_tiles = kb / 128;  // 128-byte tiles of a packed B row (256 K values for int4)
    // A as [K tiles][M rows][128 B] (3-D view, 128-byte swizzle): one copy
    // brings 8 K tiles of 16 rows.
    CUtensorMap tmA, tmB;
    {
      cuuint64_t dims[3] = {128, (cuuint64_t)M, (cuuint64_t)p.ktiles};
      cuuint64_t strides[2] = {(cuuint64_t)K, 128};
      cuuint32_t box[3] = {128, 16, 8};
      cuuint32_t estr[3] = {1, 1, 1};
      if (g_encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(A), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return GP_ERR_CUDA;
    }
    // packed B as [8-row bands][B tiles][8 rows][128 B] (4-D view, already
    // swizzled): one copy brings a stage's 1024 K values (8 tiles, or 4 of
    // int4) of a CTA's whole strip of bands.
    {
      cuuint64_t dims[4] = {128, 8, (cuuint64_t)b_tiles, (cuuint64_t)(N / 8)};
      cuuint64_t strides[3] = {128, 1024, (cuuint64_t)b_tiles * 1024};
      cuuint32_t box[4] = {128, 8, w4 ? 4u : 8u, (cuuint32_t)(p.strip / 8)};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      if (g_encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(B_packed), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return GP_ERR_CUDA;
    }
    return i8_gemm_launch(tmA, tmB, p, d->num_sms, st);
  }

  // Tile height: 256 rows (two 128-row MMAs sharing each B tile) when that
  // still gives every SM several tiles, or when K is split over a cluster
  // (few tiles); the E2M1 kernel uses 128.
  // Few 256 x 256 tiles with a long K: two pairs per tile, one per half of K.
  const bool xpair = dtype != GP_E2M1 && xpair_choice(M, N, (int)(kb / 128), d->num_sms);
  const int split = (dtype == GP_E2M1 || xpair) ? 1 : splitk_choice(M, N, kb / 128, d->num_sms);
  int bm = 128, bn = 256;
  if (dtype != GP_E2M1) {
    if (split > 1 || xpair)
      bm = 256;
    else
      tc_tile_choice(M, N, d->num_sms, &bm, &bn);
  }
  // 2-CTA pair tiles replace the single-CTA 128 x 128 and 256 x 256 tiles
  // where a tile has rows for both CTAs (0: single-CTA tiles).
  const int pair_bn = xpair ? 256 : (dtype != GP_E2M1 && split == 1) ? pair_choice(M, bm, bn) : 0;
  CUtensorMap tmA, tmC;
  const int kstep = xpair                     ? kXpairKstep
                    : pair_bn != 0              ? kPairKstep
                    : (dtype != GP_E2M1 && split == 1) ? tc_kstep(bm, bn)
                                                : 1;
  const int a_rows = pair_bn != 0 ? 128 : bm;  // rows of A per CTA
  if (kstep == 1 && !xpair) {  // (the two-pair kernel reads A through the 3-D view)
    if ((rc = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)kb, (uint64_t)M, (uint64_t)kb, 128,
                        (uint32_t)a_rows, CU_TENSOR_MAP_SWIZZLE_128B)) != GP_OK)
      return rc;
  } else {
    // A as [K tiles][M rows][128 B] (3-D view, 128-byte swizzle): one copy
    // brings `kstep` K tiles of a CTA's rows.
    cuuint64_t dims[3] = {128, (cuuint64_t)M, (cuuint64_t)(kb / 128)};
    cuuint64_t strides[2] = {(cuuint64_t)kb, 128};
    cuuint32_t box[3] = {128, (cuuint32_t)a_rows, (cuuint32_t)kstep};
    cuuint32_t estr[3] = {1, 1, 1};
    if (g_encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(A), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GP_ERR_CUDA;
  }
  if ((rc = encode_2d(&tmC, c_dtype == GP_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 64, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != GP_OK)
    return rc;
  TcParams p{};
  p.Bp = static_cast<const uint8_t*>(B_packed);
  p.status = d->status;
  p.wait_limit_ns = wait_limit_ns();
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.ktiles = (int)(kb / 128);
  p.debug_skip_load = g_debug_skip_load.exchange(0);
  p.b_constant = b_constant;
  {
    const int64_t tile_rows = (pair_bn != 0 || split > 1) ? 256 : bm;  // rows of C per tile of the chosen kernel
    p.raster_g = raster_group((M + tile_rows - 1) / tile_rows, tile_rows, kb, d->l2_bytes);
  }
  p.bias = static_cast<const float*>(bias);
  p.out_f16 = c_dtype == GP_FP16 ? 1 : 0;
  p.act = epilogue == GP_EPI_BIAS_RELU ? EPI_ACT_RELU
          : epilogue == GP_EPI_BIAS_SILU ? EPI_ACT_SILU
          : epilogue == GP_EPI_BIAS_GELU ? EPI_ACT_GELU
                                         : EPI_ACT_NONE;
  if (scale_mode == GP_SCALE_ROWCOL_F32) {
    p.sa = static_cast<const float*>(scale_a);
    p.sb = static_cast<const float*>(scale_b);
  }
  if (dtype == GP_E2M1) {
    if (N % 256 != 0) return GP_ERR_SHAPE;
    p.Bsf = p.Bp + (size_t)N * (size_t)kb;
    p.sfa = static_cast<const uint8_t*>(scale_a);
    const bool pair = mxf4_pair_choice(M);
    CUtensorMap tmB = {}, tmSFB = {};
    if (pair) {
      // packed B as [tiles][128 rows][128 B]; its scales as [bands][K steps]
      // [4][256 B] (1 KiB per band and K step, already in the TMEM copy image)
      const uint64_t bands = (uint64_t)(N / 128), ksteps = (uint64_t)(kb / 128);
      {
        cuuint64_t dims[3] = {128, 128, bands * ksteps};
        cuuint64_t strides[2] = {128, 16384};
        cuuint32_t box[3] = {128, 128, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(B_packed), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return GP_ERR_CUDA;
      }
      {
        cuuint64_t dims[4] = {256, 4, ksteps, bands};
        cuuint64_t strides[3] = {256, 1024, ksteps * 1024};
        cuuint32_t box[4] = {256, 4, 1, 2};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(p.Bsf), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return GP_ERR_CUDA;
      }
    }
    return mxf4_gemm_launch(pair, tmA, tmB, tmSFB, tmC, p, d->num_sms, st);
  }
  const int kind = dtype == GP_BF16 ? 0 : dtype == GP_E4M3 ? 1 : 2;  // 2: fp16
  if (split > 1) return splitk_gemm_launch(kind, split, tmA, tmC, p, st);
  if (pair_bn != 0) {
    // packed B as [tiles][128 rows][128 B] (3-D view, already swizzled):
    // one copy brings a CTA's pair_bn/2 rows of kPairKstep consecutive tiles
    // of a band.
    CUtensorMap tmB;
    cuuint64_t dims[3] = {128, 128, (cuuint64_t)(N / 128) * (cuuint64_t)(kb / 128)};
    cuuint64_t strides[2] = {128, 16384};
    cuuint32_t box[3] = {128, (cuuint32_t)(pair_bn / 2), (cuuint32_t)kstep};
    cuuint32_t estr[3] = {1, 1, 1};
    if (g_encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(B_packed), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GP_ERR_CUDA;
    if (xpair) return xpair_gemm_launch(kind, tmA, tmB, tmC, p, st);
    return pair_gemm_launch(kind, pair_bn, tmA, tmB, tmC, p, d->num_sms, st);
  }
  return tc_gemm_launch(kind, bm, bn, tmA, tmC, p, d->num_sms, st);
}

int gemm_last_device_status(void* stream) {
  DeviceInfo* d = nullptr;
  int rc = device_info(&d);
  if (rc != GP_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GP_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GP_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GP_ERR_CUDA;
    return (word & ST_BAD_LAUNCH) ? GP_ERR_DEVICE_CHECK : GP_ERR_DEVICE_TIMEOUT;
  }
  return GP_OK;
}

int gemm_quantize_a(const void* X, int x_dtype, int64_t M, int64_t K, int q_dtype, void* A_out, void* scales_out,
                    void* stream) {
  if ((x_dtype != GP_FP32 && x_dtype != GP_BF16) || (q_dtype != GP_E4M3 && q_dtype != GP_E2M1))
    return GP_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || K % 32 != 0) return GP_ERR_SHAPE;
  if (M == 0 || K == 0) return GP_OK;
  if (X == nullptr || A_out == nullptr || scales_out == nullptr) return GP_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(A_out) || !aligned16(scales_out)) return GP_ERR_ALIGNMENT;
  DeviceInfo* d = nullptr;
  int rc = device_info(&d);
  if (rc != GP_OK) return rc;
  return quant_launch(X, x_dtype == GP_BF16, M, K, q_dtype == GP_E2M1, A_out, scales_out, d->num_sms, d->status,
                      wait_limit_ns(), static_cast<cudaStream_t>(stream));
}

// Test hook: the next tcgen05 GEMM launch skips the producer's `index`-th
// stage load (1-based), so its bounded waits time out.  0 disables it.
int gemm_debug_skip_load(int index) {
  if (index < 0) return GP_ERR_INVALID_ARG;
  g_debug_skip_load.store(index);
  return GP_OK;
}

}  // extern "C"
