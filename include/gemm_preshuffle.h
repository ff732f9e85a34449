/*
 * gemm_preshuffle.h -- C ABI of the GB300 (sm_103a) preshuffle GEMM library.
 *
 *   C[M,N] = A[M,K] . B[N,K]^T
 *
 * "GEMM Optimization Guide", section 1.1: the product and its tiling.
 * Section 12 (B matrix preshuffle layout): B is permuted once, offline, into
 * a layout that the kernel's loads copy without further shuffling.  This
 * library uses its own layout for that step, shaped for TMA and tcgen05.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA global-memory pointers that the caller owns.
 *     The library never frees them and never keeps them after a call returns.
 *   - `stream` is a cudaStream_t passed as void*.  NULL means the legacy
 *     default stream.
 *   - Calls are asynchronous with respect to the host and ordered on `stream`.
 *     The GEMM and quantiser kernels are launched with programmatic
 *     dependent launch: a kernel may become resident while the previous
 *     kernel on the stream still runs, but it reads and writes the caller's
 *     buffers only after that kernel has finished.  The two exceptions are
 *     opt-in: GP_RUN_B_CONSTANT and GP_RUN_INDEPENDENT (gemm_run_ex).
 *   - Argument errors are detected on the host before anything is launched.
 *     The call then returns a nonzero gp_status and leaves all buffers
 *     untouched.
 *   - Device-side timeouts of the bounded waits inside the GEMM and
 *     quantiser kernels set a sticky status word.  gemm_last_device_status()
 *     reads and clears it.
 *   - Matrices are row-major and densely packed (row pitch = K elements for
 *     A and B, N elements for C).
 *   - Every device pointer must be 16-byte aligned.
 *   - Thread safety: calls from several host threads are safe.  Each call
 *     keeps its state on the stack, apart from a per-device table of SM
 *     counts and function attributes, which is written once under a lock.
 */
#ifndef GEMM_PRESHUFFLE_H
#define GEMM_PRESHUFFLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum gp_status {
  GP_OK = 0,
  GP_ERR_INVALID_ARG = 1,     /* null pointer where one is required, bad enum */
  GP_ERR_UNSUPPORTED = 2,     /* dtype / scale-mode / output combination not offered */
  GP_ERR_SHAPE = 3,           /* dimension rule violated (see gemm_run) */
  GP_ERR_ALIGNMENT = 4,       /* a pointer is not 16-byte aligned */
  GP_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed */
  GP_ERR_DEVICE_TIMEOUT = 6,  /* a bounded in-kernel wait gave up (see gemm_last_device_status) */
  GP_ERR_DEVICE_CHECK = 7     /* a kernel's launch self-check failed (see gemm_last_device_status) */
} gp_status;

/* Element types.  E4M3 is OCP E4M3FN.  E2M1 packs two codes per byte, with
 * the even-k element in the low nibble. */
typedef enum gp_dtype {
  GP_BF16 = 0,
  GP_E4M3 = 1,
  GP_INT8 = 2,
  GP_E2M1 = 3,
  GP_INT32 = 4,
  GP_FP16 = 5,                /* IEEE binary16 */
  GP_FP32 = 6,                /* IEEE binary32 (quantiser input only) */
  GP_W4A8 = 7                 /* int4 B (two's complement nibbles, two per byte, even k
                                 low) with int8 A; "GEMM Optimization Guide" section 8.2
                                 counts N*K//2 bytes for such a B */
} gp_dtype;

/* How operand scales enter the product. */
typedef enum gp_scale_mode {
  GP_SCALE_NONE = 0,          /* C = sum_k A*B */
  GP_SCALE_ROWCOL_F32 = 1,    /* C[m,n] = (sum_k A*B) * scale_a[m] * scale_b[n], fp32 scales.
                                 "GEMM Optimization Guide" section 7.1: the epilogue forms
                                 acc * scale_a * scale_b; section 8.2 counts (M+N) fp32 scales. */
  GP_SCALE_BLOCK32_UE8M0 = 2  /* MX block scaling: one UE8M0 exponent per 32 consecutive K
                                 elements of each row of A and of B (section 8.2, MXFP4 bytes):
                                 C = sum_j 2^(ea[m,j]-127) 2^(eb[n,j]-127) sum_{k in block j} A*B */
} gp_scale_mode;

/*
 * Size in bytes of the packed B buffer for a [N, K] operand of `dtype`.
 * The packed layout holds the same bytes as B, followed by B's packed block
 * scales for E2M1, with no padding.
 *
 * Shape rules: N % 128 == 0 and K*element_bits/8 % 128 == 0.  For the
 * element types that means K % 128 (E4M3, INT8), K % 64 (BF16, FP16) and
 * K % 256 (E2M1, and W4A8, whose packed B holds the int4 weights).
 * Returns GP_ERR_SHAPE otherwise.  Host-only call.
 */
int gemm_packed_b_bytes(int dtype, int64_t N, int64_t K, size_t* bytes_out);

/*
 * The offline preshuffle of B ("GEMM Optimization Guide" section 12).
 *
 * B         : device, [N, K] row-major in `dtype` (E2M1: [N, K/2] bytes).
 * B_scales  : device, UE8M0 [N, K/32] row-major, required for E2M1 (NULL otherwise).
 * B_packed  : device, gemm_packed_b_bytes() bytes, written entirely.
 *
 * Layout of the packed buffer (a bijection of B's bytes):
 *   - B's bytes are cut into tiles of R rows x 128 bytes, with R = 128 for
 *     BF16, FP16, E4M3 and E2M1 and R = 8 for INT8 and W4A8.  The tile of (row band tn,
 *     byte column tk) is the R*128-byte block with index tn*(Kb/128)+tk,
 *     where Kb = row bytes.
 *   - INT8 bytes are stored in offset binary: b XOR 0x80, i.e. b + 128 as
 *     an unsigned byte.  W4A8's int4 B also uses 8-row bands; each 32-bit
 *     word of a row (8 K values, two's complement nibbles at bits 4k) is
 *     stored with every nibble in offset binary (b + 8) and k0..k7 at bits
 *     0, 16, 4, 20, 8, 24, 12, 28.
 *   - Inside a tile, row r sits at r*128.  Its 16-byte chunk c is stored at
 *     chunk slot c ^ (r % 8).  That is the 128-byte-swizzled K-major image
 *     that tcgen05 and TMA use, so one bulk copy moves a 128-row tile into
 *     shared memory ready for the MMA; the INT8 kernel's TMA copies take
 *     any run of whole 8-row bands.
 *   - For E2M1, the block scales follow the data.  They are packed per
 *     (row band, 128-byte K tile) in two 512-byte groups of four K blocks.
 *     In a group, the byte for (row r, block j) is at
 *     (r%32)*16 + (r/32)*4 + j%4.
 * The call runs one device kernel on `stream`.
 */
int gemm_preshuffle_b(const void* B, const void* B_scales, int dtype, int64_t N, int64_t K,
                      void* B_packed, void* stream);

/*
 * The inverse of gemm_preshuffle_b.  It rebuilds B (and, for E2M1, B_scales)
 * from a packed buffer, for round-trip checks.  B_scales_out may be NULL
 * except for E2M1.
 */
int gemm_unpack_b(const void* B_packed, int dtype, int64_t N, int64_t K, void* B_out,
                  void* B_scales_out, void* stream);

/*
 * C = A . B^T with B pre-packed ("GEMM Optimization Guide" sections 1-7).
 *
 * A        : device, [M, K] row-major in `dtype` (E2M1: [M, K/2] bytes).
 * B_packed : device, output of gemm_preshuffle_b for the same dtype, N, K.
 * scale_a, scale_b : device, per `scale_mode`.  NULL for GP_SCALE_NONE.
 *            ROWCOL_F32: fp32 [M] and fp32 [N].
 *            BLOCK32_UE8M0: scale_a is UE8M0 [M, K/32] row-major (plain,
 *            not packed), and scale_b must be NULL because B's scales live
 *            in B_packed.
 * C        : device, [M, N] row-major in `c_dtype`, written entirely.
 *
 * Supported (dtype, scale_mode, c_dtype) combinations, where FOUT is
 * GP_BF16 or GP_FP16:
 *   (GP_BF16, GP_SCALE_NONE,          FOUT)      fp32 accumulation in TMEM
 *   (GP_FP16, GP_SCALE_NONE,          FOUT)      fp32 accumulation in TMEM
 *   (GP_E4M3, GP_SCALE_ROWCOL_F32,    FOUT)      fp32 accumulation, scales in epilogue
 *   (GP_E4M3, GP_SCALE_NONE,          FOUT)
 *   (GP_E2M1, GP_SCALE_BLOCK32_UE8M0, FOUT)      block scales applied inside the MMA
 *   (GP_INT8, GP_SCALE_NONE,          GP_INT32)  exact integer result
 *   (GP_W4A8, GP_SCALE_NONE,          GP_INT32)  exact integer result; A is int8 [M, K],
 *                                                B int4 [N, K/2] bytes (packed as W4A8)
 * Other combinations return GP_ERR_UNSUPPORTED.
 *
 * Shape rules: M >= 1 (any value), N and K as for gemm_packed_b_bytes, and
 * M, N, K < 2^31.  (The INT8/W4A8 kernel is built for small M; past 65535
 * groups of 16 rows it is launched once per 65535 groups.)  E2M1 also needs N % 256 == 0 (its tiles are 256 wide).
 * For INT8 the exact result must fit int32, which holds for every input
 * when K < 131072, i.e. K <= 130944 (W4A8: K < 2097152, i.e. K <= 2096896):
 * (-128) * (-128) * 131072 is already 2^31.
 * Float outputs are rounded to nearest-even from the fp32 value (an fp16
 * output saturates to infinity beyond 65504, as IEEE rounding does).
 * The call launches one kernel and allocates no memory.  K == 0 writes
 * zeros to C with an async memset.  M == 0 or N == 0 is a no-op.
 */
int gemm_run(const void* A, const void* B_packed, int dtype, int64_t M, int64_t N, int64_t K,
             int scale_mode, const void* scale_a, const void* scale_b, void* C, int c_dtype,
             void* stream);

/* Fused epilogues of the float-output products ("Kernel Tuning Guide",
 * section 6, Epilogue Strategies, names "none", "bias", "bias_relu",
 * "bias_silu" and "bias_gelu").  After the scales, v = acc * scale_a[m] *
 * scale_b[n] + bias[n] with bias fp32 [N], then the activation: ReLU
 * max(v, 0); SiLU v / (1 + e^-v); GELU 0.5 v (1 + erf(v / sqrt 2)) (the
 * exact form).  The result is rounded to the float c_dtype (bf16 or fp16). */
typedef enum gp_epilogue {
  GP_EPI_NONE = 0,
  GP_EPI_BIAS = 1,
  GP_EPI_BIAS_RELU = 2,
  GP_EPI_BIAS_SILU = 3,
  GP_EPI_BIAS_GELU = 4
} gp_epilogue;

/* Flags of gemm_run_ex. */
typedef enum gp_run_flags {
  GP_RUN_DEFAULT = 0,
  /* B_packed holds constant weights: nothing that may still be running on
   * the GPU when the call is made writes it (pack the weights once and
   * synchronise, as at model load).  The kernel may then start copying B
   * into shared memory before the kernel that precedes it on `stream` has
   * finished, which hides its pipeline start behind that kernel's tail.  A,
   * the scales and C are still touched only after the preceding kernel
   * completes.  Breaking the condition gives undefined results. */
  GP_RUN_B_CONSTANT = 1,
  /* The call is independent of the GPU work before it on `stream`: nothing
   * that may still be running when the call is made writes A, B_packed,
   * the scales or bias, or reads or writes C (for instance a run of GEMMs on
   * weights of their own, into outputs of their own, whose activations were
   * produced before the run).  The weight-streaming INT8/W4A8 kernel then
   * runs its whole body alongside the preceding kernel and waits for that
   * kernel only before it exits, so its completion still follows the
   * completion of everything before it and work queued after the call sees
   * every earlier result.  The tcgen05 kernels take this flag as
   * GP_RUN_B_CONSTANT.  Implies GP_RUN_B_CONSTANT; breaking the condition
   * gives undefined results. */
  GP_RUN_INDEPENDENT = 2
} gp_run_flags;

/*
 * gemm_run with a fused epilogue and flags; gemm_run is gemm_run_ex with
 * GP_EPI_NONE, bias NULL and GP_RUN_DEFAULT.
 *
 * epilogue : a gp_epilogue.  Any value but GP_EPI_NONE needs a float
 *            c_dtype (GP_BF16 or GP_FP16; else GP_ERR_UNSUPPORTED: the
 *            INT8 product keeps its exact int32 output).
 * bias     : device, fp32 [N], 16-byte aligned; required for every epilogue
 *            but GP_EPI_NONE, and NULL with it (else GP_ERR_INVALID_ARG).
 * flags    : a bitwise OR of gp_run_flags.  Unknown bits return
 *            GP_ERR_INVALID_ARG before any launch.  GP_RUN_B_CONSTANT and
 *            GP_RUN_INDEPENDENT are scheduling options of this library: the
 *            method itself only assumes that the packed weights are
 *            produced once, offline ("GEMM Optimization Guide" section 12).
 * The other arguments are as for gemm_run.  With K == 0 the product is
 * zero, so every row of C is act(bias[n]) (a broadcast kernel).
 */
int gemm_run_ex(const void* A, const void* B_packed, int dtype, int64_t M, int64_t N, int64_t K,
                int scale_mode, const void* scale_a, const void* scale_b, int epilogue,
                const void* bias, void* C, int c_dtype, unsigned flags, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  The word is set when a bounded wait in a GEMM
 * or quantiser kernel times out, or when a kernel's check of its own launch shape against
 * its arguments fails (the kernel then returns before touching memory).
 * Returns GP_OK, GP_ERR_DEVICE_TIMEOUT, GP_ERR_DEVICE_CHECK or GP_ERR_CUDA.
 */
int gemm_last_device_status(void* stream);

/*
 * The activation quantiser in front of the GEMM: the operand recipes of the
 * FP8 and MXFP4 products ("GEMM Optimization Guide" section 8.2: per-token
 * fp32 scales; one UE8M0 byte per 32 K-elements).
 *
 * X          : device, [M, K] row-major, x_dtype GP_FP32 or GP_BF16.
 * q_dtype    : GP_E4M3 or GP_E2M1.
 * A_out      : device.  E4M3: uint8 codes [M, K].  E2M1: uint8 [M, K/2],
 *              two codes per byte, even k in the low nibble.  Ready to be
 *              gemm_run's A.
 * scales_out : device.  E4M3: fp32 [M], s[m] = amax_k |X[m,k]| / 448 (1 for
 *              an all-zero row), with codes E4M3FN(X / s).  E2M1: UE8M0
 *              [M, K/32], e + 127 where e is the smallest integer with
 *              amax over the block <= 6 * 2^e (0 for an all-zero block), with
 *              codes E2M1(X * 2^-e).  Ready to be gemm_run's scale_a.
 * Codes round to nearest even and saturate (+-448, +-6).  The divisions
 * are IEEE fp32, so the result is bit-exact for given inputs.  NaN or
 * infinite inputs are not supported.
 * Shape rules: K % 32 == 0; M, K < 2^31.  M == 0 or K == 0 is a no-op.
 * Pointers must be 16-byte aligned (GP_ERR_ALIGNMENT).  One kernel on
 * `stream`; nothing is allocated.  Its waits on its own row copies are
 * bounded: a timeout sets the device status word (gemm_last_device_status).
 * This step precedes the method's GEMM; the pages do it on the host for
 * their inputs.
 */
int gemm_quantize_a(const void* X, int x_dtype, int64_t M, int64_t K, int q_dtype, void* A_out,
                    void* scales_out, void* stream);

/* Static, human-readable name of a gp_status value. */
const char* gemm_status_string(int status);

/*
 * Fault-injection hook for tests of the bounded waits; it has no
 * counterpart in the method.  The next GEMM launched by gemm_run (any of
 * its kernels: tile, split-K, MXFP4, INT8/W4A8) skips its producer's
 * `index`-th shared-memory stage load (1-based).  For INT8/W4A8 the B
 * load of that stage and of every later stage is skipped.
 * The waits for that stage then time out after the wait limit, which
 * defaults to 2 s and is overridden by the environment variable
 * GP_WAIT_LIMIT_MS, read once per process.
 *
 * When the wait times out, the kernel drains its in-flight copies, frees
 * any tensor memory and exits.  The library's status word is set, and
 * gemm_last_device_status() reports GP_ERR_DEVICE_TIMEOUT.  The hook
 * disarms itself after one launch.  index = 0 disarms it.  Host-only.
 */
int gemm_debug_skip_load(int index);

#ifdef __cplusplus
}
#endif
#endif /* GEMM_PRESHUFFLE_H */
