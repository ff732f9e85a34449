// Tensor-pipe rate of each tcgen05.mma kind the library uses, measured on the
// GPU at hand: the denominators of the tensor rooflines for FP8 and MXFP4,
// which otherwise rest on nominal ratios to the measured bf16 rate.
//
// Every SM runs one CTA (or one CTA of a 2-CTA cluster) whose single issuing
// thread streams back-to-back MMAs over one 128-byte K tile of fixed
// shared-memory operands (M = 128 or 256 over a pair, N = 256, four
// instructions a K tile), accumulating into tensor memory.  No global memory
// is touched besides two timestamps a CTA, so the loop shows the tensor
// pipe's own rate.  The final commit is awaited with a bounded wait.
//
// Usage: mma_rate [iterations = 20000] [repetitions = 2]; one JSON line per
// kind and form: {"kind", "form", "tflops", "tflops_per_sm", "ms", "ok"}.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include <cuda_runtime.h>

#include "../csrc/ptx.cuh"

using namespace gp;

namespace {

// kind: 0 bf16, 2 fp16 (kind::f16), 1 e4m3 (kind::f8f6f4), 3 e2m1 with UE8M0
// scales per 32 (kind::mxf4.block_scale.scale_vec::2X)
constexpr int kSmem = 200 * 1024;  // one CTA an SM

// scale-factor block for tcgen05.cp: 32 rows x 16 bytes, no swizzle
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

template <int KIND, bool PAIR>
__global__ void __launch_bounds__(128, 1) mma_loop(int iters, unsigned long long* t_out, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int B_ROWS = PAIR ? 128 : 256;  // this CTA's rows of B
  uint8_t* s_a = base;                      // 128 rows x 128 B
  uint8_t* s_b = base + 16384;              // B_ROWS rows x 128 B
  uint8_t* s_sf = s_b + B_ROWS * 128;       // 4 KiB of scale bytes, each 2^0
  uint64_t* bar = reinterpret_cast<uint64_t*>(s_sf + 4096);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int ab_words = (16384 + B_ROWS * 128) / 4;
  for (int i = threadIdx.x; i < ab_words; i += blockDim.x)
    reinterpret_cast<uint32_t*>(base)[i] = 0x3C3C3C3Cu ^ ((uint32_t)i * 2654435761u & 0x07070707u);
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) reinterpret_cast<uint32_t*>(s_sf)[i] = 0x7F7F7F7Fu;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    if constexpr (PAIR)
      tmem_alloc_pair<512>(slot);
    else
      tmem_alloc<512>(slot);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *slot;
  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(s_a), b0 = smem_u32(s_b);
    // scale slots beside the 256-column accumulator: A at 256 (4 columns an
    // atom), B at 264 (8 columns an atom, two 128-row bands)
    if constexpr (KIND == 3) {
      for (int at = 0; at < 2; ++at) {
        const uint64_t da = sf_desc(smem_u32(s_sf) + at * 512);
        if constexpr (PAIR)
          tmem_cp_32x128b_warpx4_pair(tbase + 256 + at * 4, da);
        else
          tmem_cp_32x128b_warpx4(tbase + 256 + at * 4, da);
        for (int j = 0; j < 2; ++j) {
          const uint64_t db = sf_desc(smem_u32(s_sf) + 1024 + j * 1024 + at * 512);
          if constexpr (PAIR)
            tmem_cp_32x128b_warpx4_pair(tbase + 264 + at * 8 + j * 4, db);
          else
            tmem_cp_32x128b_warpx4(tbase + 264 + at * 8 + j * 4, db);
        }
      }
    }
    constexpr uint32_t M = PAIR ? 256 : 128;
    const unsigned long long t0 = globaltimer();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t acc = (it | k) != 0 ? 1u : 0u;
        const uint64_t da = smem_desc_sw128(a0 + 32 * k), db = smem_desc_sw128(b0 + 32 * k);
        if constexpr (KIND == 3) {
          const uint32_t at = (uint32_t)(k >> 1), id = (uint32_t)(k & 1) * 2;
          if constexpr (PAIR)
            umma_mxf4_pair(tbase, da, db, idesc_mxf4(M, 256, id, id), tbase + 256 + at * 4, tbase + 264 + at * 8,
                           acc);
          else
            umma_mxf4(tbase, da, db, idesc_mxf4(M, 256, id, id), tbase + 256 + at * 4, tbase + 264 + at * 8, acc);
        } else {
          constexpr uint32_t fmt = KIND == 0 ? 1u : 0u;  // bf16, or fp16 / e4m3 (0)
          if constexpr (PAIR)
            umma_pair<KIND>(tbase, da, db, idesc_dense(fmt, fmt, M, 256), acc);
          else
            umma<KIND>(tbase, da, db, idesc_dense(fmt, fmt, M, 256), acc);
        }
      }
    }
    if constexpr (PAIR)
      umma_commit_pair(bar, 0x3);
    else
      umma_commit(bar);
    volatile int never = 0;
    const bool ok = wait_bounded(bar, 0, &never, status, 1u, 5000000000ull);
    const unsigned long long t1 = globaltimer();
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    t_out[2 * unit] = t0;
    t_out[2 * unit + 1] = ok ? t1 : 0ull;
  }
  if (PAIR && rank == 1 && threadIdx.x == 0) {
    volatile int never = 0;
    wait_bounded(bar, 0, &never, status, 2u, 6000000000ull);  // the pair's MMAs are complete
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair<512>(tbase);
    else
      tmem_dealloc<512>(tbase);
  }
}

template <int KIND, bool PAIR>
void run(const char* kind, double k_elems, int iters, int reps, int sms) {
  auto kern = mma_loop<KIND, PAIR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) {
    printf("{\"kind\": \"%s\", \"form\": \"%s\", \"ok\": false}\n", kind, PAIR ? "cta_group::2" : "cta_group::1");
    return;
  }
  const int units = PAIR ? sms / 2 : sms;
  unsigned long long* d_t = nullptr;
  uint32_t* d_st = nullptr;
  cudaMalloc(&d_t, sizeof(unsigned long long) * 2 * units);
  cudaMalloc(&d_st, 4);
  cudaMemset(d_st, 0, 4);
  std::vector<unsigned long long> h(2 * units);
  const double m = PAIR ? 256.0 : 128.0;
  const double flop_per_unit = 2.0 * m * 256.0 * k_elems * 4.0 * iters;
  for (int r = 0; r < reps; ++r) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(PAIR ? 2 * units : units);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, iters, d_t, d_st);
    const cudaError_t se = cudaDeviceSynchronize();
    cudaMemcpy(h.data(), d_t, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    uint32_t st = 0;
    cudaMemcpy(&st, d_st, 4, cudaMemcpyDeviceToHost);
    unsigned long long lo = ~0ull, hi = 0;
    double sum = 0;
    int good = 0;
    for (int i = 0; i < units; ++i) {
      if (h[2 * i + 1] == 0) continue;
      lo = std::min(lo, h[2 * i]);
      hi = std::max(hi, h[2 * i + 1]);
      sum += (double)(h[2 * i + 1] - h[2 * i]);
      ++good;
    }
    const bool ok = le == cudaSuccess && se == cudaSuccess && st == 0 && good == units;
    const double span_s = good > 0 ? (double)(hi - lo) * 1e-9 : 1.0;
    const double per_sm = good > 0 ? flop_per_unit / (sum / good * 1e-9) / 1e12 / (PAIR ? 2.0 : 1.0) : 0.0;
    printf("{\"kind\": \"%s\", \"form\": \"%s\", \"tflops\": %.1f, \"tflops_per_sm\": %.3f, \"ms\": %.3f, "
           "\"ok\": %s}\n",
           kind, PAIR ? "cta_group::2" : "cta_group::1", flop_per_unit * good / span_s / 1e12, per_sm, span_s * 1e3,
           ok ? "true" : "false");
    fflush(stdout);
  }
  cudaFree(d_t);
  cudaFree(d_st);
}

}  // namespace

int main(int argc, char** argv) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 2) {
    printf("{\"ok\": false, \"error\": \"no device\"}\n");
    return 1;
  }
  const int iters = argc > 1 ? std::max(1, atoi(argv[1])) : 20000;
  const int reps = argc > 2 ? std::max(1, atoi(argv[2])) : 2;
  // K elements per instruction: 16 (16-bit), 32 (e4m3), 64 (e2m1)
  run<0, false>("bf16", 16, iters, reps, sms);
  run<2, false>("fp16", 16, iters, reps, sms);
  run<1, false>("e4m3", 32, iters, reps, sms);
  run<3, false>("e2m1", 64, iters, reps, sms);
  run<0, true>("bf16", 16, iters, reps, sms);
  run<1, true>("e4m3", 32, iters, reps, sms);
  run<3, true>("e2m1", 64, iters, reps, sms);
  return 0;
}
