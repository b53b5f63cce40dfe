/*
 * gemm.h -- C ABI of libgemm: dense C = A*B on one GB300 GPU (sm_103a).
 *
 * The operation.  With A of size M x K, B of size K x N and C of size M x N,
 *     C_ij = sum over k = 0 .. K-1 of A_ik * B_kj
 * ("Shared Memory Tiling for Matrix Multiplication", opening formula).  All
 * three matrices are dense and row-major with no leading-dimension argument:
 * A_ik is A[i*K + k], B_kj is B[k*N + j], C_ij is C[i*N + j] ("Matrix
 * Multiplication -- Naive to Tiled", section 02).  C is overwritten, as that
 * page's kernels store the finished sum; it is never read.
 *
 * Argument order (M, K, N) follows the kernel signature of that same section.
 *
 * Every pointer is a DEVICE pointer on the calling thread's current CUDA
 * device; the caller owns all buffers and the stream, and the library frees
 * nothing it did not allocate.  Every call is asynchronous: it validates its
 * arguments on the host, enqueues its kernels on `stream` and returns.  Device
 * errors of an earlier call surface through gemm_debug_status() or the
 * caller's own synchronisation.  No call exits the process or traps the GPU.
 *
 * `stream` is a cudaStream_t (the pointer type is declared here so this header
 * needs no CUDA header); NULL means the legacy default stream.
 *
 * Environment (testing and tuning only; read once per process): with
 * GEMM_FORCE_CONFIG=single_cta the tensor-core modes use the 1-SM kernel even
 * where 2-SM clusters fit; =b_boxes_2d makes them load B by 2-D boxes per
 * column block even where the atom-ordered 4-D form applies (same results,
 * bit for bit); =ffma_small / =ffma_tiles128 make every GEMM_FP32 product
 * take the 32 x 32-tile or the 128 x 128-tile FFMA kernel instead of the one
 * chosen by shape; =ffma_no_stream keeps GEMM_FP32 products of a quarter of a
 * wave to two waves of tiles off the stream-K form.  Results stay within each mode's
 * tolerance.
 */
#ifndef LIBGEMM_GEMM_H
#define LIBGEMM_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the type behind cudaStream_t */

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

/* precision_mode values */
enum gemm_mode {
    /* A, B: const float*.  Exact binary32 arithmetic on the CUDA cores: every
     * product-accumulate is one fused multiply-add rounded to nearest, k
     * ascending for each C_ij.  When the output tiles do not fill the GPU
     * and K is long, the library cuts K into consecutive ranges, runs the
     * chain over each range and adds the range sums in range order (binary32
     * adds): the same result on every run of the same shape. */
    GEMM_FP32 = 0,
    /* A, B: const float*.  Tensor cores (tcgen05, kind::tf32): the inputs are
     * read as TF32 (sign, 8-bit exponent, top 10 fraction bits of each
     * binary32), products are accumulated in binary32. */
    GEMM_TF32 = 1,
    /* A, B: const uint16_t* holding bfloat16 values (the caller rounds its
     * data to bfloat16).  Tensor cores (tcgen05, kind::f16 with BF16
     * inputs), binary32 accumulation. */
    GEMM_BF16 = 2,
    /* A, B: const uint16_t* holding IEEE binary16 values.  Tensor cores
     * (tcgen05, kind::f16 with F16 inputs), binary32 accumulation -- the
     * FP16-input, FP32-accumulate product the first page's "Further
     * Optimisation Ideas" names for tensor cores. */
    GEMM_FP16 = 3,
    /* A, B: const float*.  The library rounds them to bfloat16 (to nearest,
     * ties to even) in a conversion pass, then multiplies as GEMM_BF16:
     * BF16 tensor-core speed for float data, at BF16 input precision.  The
     * result equals GEMM_BF16 on the caller-rounded operands, bit for bit. */
    GEMM_FP32_VIA_BF16 = 4,
    /* A, B: const float*.  As GEMM_TF32, but the library first rounds each
     * input to the nearest TF32 value (ties away from zero) in a conversion
     * pass, instead of letting the tensor cores drop the 13 low fraction
     * bits: the rounding errors of the inputs then have no sign bias, at the
     * cost of the pass (scratch for the rounded copies of A and B).  The
     * result equals GEMM_TF32 on the caller-rounded operands, bit for bit. */
    GEMM_TF32_RN = 5
};

/* Status codes returned by every entry point (0 = success). */
enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* NULL pointer with a non-empty matrix, negative
                                        dimension, unknown mode, C overlapping A or B,
                                        or a size whose element count overflows int64 */
    GEMM_ERR_MISALIGNED = 2,         /* pointer not aligned to its element size
                                        (4 bytes for float, 2 for bfloat16/binary16) */
    GEMM_ERR_CUDA = 3,               /* a CUDA runtime call or kernel launch failed */
    GEMM_ERR_NO_MEMORY = 4,          /* the stream-ordered scratch allocation failed */
    GEMM_ERR_UNSUPPORTED_DEVICE = 5, /* the current device is not compute capability 10.3 */
    GEMM_ERR_TIMEOUT = 6,            /* a bounded wait inside a kernel expired; the kernel
                                        stopped early and its output is not valid */
    GEMM_ERR_SCRATCH_LIMIT = 7,      /* gemm_tf32_noalloc: the product needs more scratch
                                        than GEMM_NOALLOC_SCRATCH_BYTES */
    GEMM_ERR_BOUNDS = 8              /* debug build only (gemm_debug_build() == 1): a kernel
                                        computed a global-memory access outside the buffer
                                        it belongs to; the access was skipped and the
                                        output is not valid */
};

/*
 * C = A*B.
 *   A               device pointer to M*K elements (float; bfloat16 in GEMM_BF16;
 *                   binary16 in GEMM_FP16)
 *   B               device pointer to K*N elements (same element type as A)
 *   C               device pointer to M*N floats; overwritten; must not overlap A or B
 *   M, K, N         dimensions, each >= 0.  M == 0 or N == 0: nothing is done.
 *                   K == 0: C is set to 0 (the empty sum).
 *   precision_mode  one of enum gemm_mode
 *   stream          stream to enqueue on
 * GEMM_FP32_VIA_BF16 and GEMM_TF32_RN take scratch for the rounded copies of A
 * and B, from the same stream-ordered allocator.
 * Any alignment of element size or more is accepted.  When a tensor-core mode
 * meets a row stride that is not a multiple of 16 bytes, or a base address
 * that is not 16-byte aligned, the operand is first copied into a scratch
 * buffer with a padded row stride; that buffer is taken from and returned to
 * CUDA's stream-ordered allocator on `stream` inside the call.  GEMM_FP32
 * does the same for B (K * roundup(N, 4) floats) when B's rows are not
 * 16-byte aligned and M >= 1024, so that B can be read 16 bytes at a time;
 * the K-split forms of both paths take workspace from the same allocator.
 * Returns GEMM_OK or an enum gemm_status code; on an error nothing is enqueued.
 */
GEMM_API int gemm(const void* A, const void* B, float* C, int64_t M, int64_t K, int64_t N,
         int precision_mode, struct CUstream_st* stream);

/*
 * C = alpha*A*B + beta*C -- the generalised product of the cuBLAS call that
 * "Matrix Multiplication -- Naive to Tiled" (section 07, Further Optimisation
 * Ideas) uses as its yardstick, for the same row-major operands as gemm().
 *   alpha, beta     binary32 scalars (host values)
 *   other arguments as for gemm(); C is read as well as written when beta != 0
 * Each C_ij is computed from the mode's sum acc_ij as fma(beta, C_ij, alpha *
 * acc_ij), the product alpha * acc_ij rounded to binary32 first and the fused
 * multiply-add rounded once.  Conventions of the BLAS, where the page is
 * silent:
 *   beta == 0       C is not read (NaN or garbage in C does not propagate);
 *                   each C_ij := alpha * acc_ij.
 *   alpha == 0, or K == 0   A and B are not read and no product is formed;
 *                   C := beta * C (each element rounded once), C := 0 when
 *                   beta == 0 as well, and nothing is enqueued when beta == 1.
 *   alpha == 1, beta == 0   identical to gemm(), bit for bit.
 * Validation, status codes, scratch use and asynchrony are those of gemm().
 */
GEMM_API int gemm_ex(const void* A, const void* B, float* C, int64_t M, int64_t K, int64_t N,
                     float alpha, float beta, int precision_mode, struct CUstream_st* stream);

/* Static, human-readable name of a status code ("unknown status" otherwise). */
GEMM_API const char* gemm_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word, which kernels set when a bounded wait expires, and, in the debug
 * build, the bounds-check flags.  Returns GEMM_OK, GEMM_ERR_TIMEOUT,
 * GEMM_ERR_BOUNDS (debug build; a timeout is reported first when both
 * happened), or GEMM_ERR_CUDA if the synchronisation itself failed.
 */
GEMM_API int gemm_debug_status(struct CUstream_st* stream);

/*
 * 1 when this library was built with device-side bounds checks (compiled
 * with GEMM_DEBUG: every kernel checks each global access against the extent
 * of the buffer it belongs to, skips one that falls outside and records it
 * for gemm_debug_status), 0 for the release build, whose kernels carry no
 * checks.  The checks stand in for a memory checker where none can run.
 */
GEMM_API int gemm_debug_build(void);

/* Library version as major*10000 + minor*100 + patch. */
GEMM_API int gemm_version(void);

/*
 * Number of kernels this library has launched in this process, all devices
 * and streams together.  Lets a benchmark count the launches in a timed
 * region.
 */
GEMM_API int64_t gemm_launch_count(void);

/*
 * Self-test of the bounded wait used by the tensor-core kernel's pipeline:
 * launches one block that waits on a barrier nothing will ever complete,
 * giving up after `timeout_ns` nanoseconds (clamped to 1 us .. 2 s), and
 * synchronises.  Returns GEMM_ERR_TIMEOUT when the wait expired and was
 * reported as it should be, GEMM_OK if it was not (a defect), or a launch
 * error.  Clears the error word before returning.  The GPU stays usable.
 */
GEMM_API int gemm_selftest_bounded_wait(int64_t timeout_ns, struct CUstream_st* stream);

/*
 * gemm_tf32_noalloc -- the GEMM_TF32 product without allocating device memory.
 *
 * The pages have no counterpart for this entry point; it is a service of this
 * library.  gemm() in GEMM_TF32 sometimes needs scratch memory -- a copy of A
 * or B with 16-byte row strides when TMA cannot read them in place (K or N
 * not a multiple of 4, or a base not 16-byte aligned), and the workspace of
 * a K split (products with few output tiles and a long K, or a partial last
 * round of tiles, e.g. 4096^3) -- and takes it from CUDA's stream-ordered
 * allocator.  Some callers cannot allow that: a host application that has
 * reserved the device memory for its own pool, so an allocation would fail
 * or eat into its budget; or a latency-critical loop where an allocation may
 * stall or fail at a bad moment.  This entry point uses instead one static
 * device buffer of GEMM_NOALLOC_SCRATCH_BYTES, compiled into the library: it
 * never calls cudaMalloc, cudaMallocAsync, cudaFree or any allocating
 * routine.
 *
 * Arguments and results are those of gemm() with precision_mode GEMM_TF32:
 * A, B, C device pointers (float, 4-byte aligned), row-major, C overwritten,
 * asynchronous on `stream`.  The product is planned exactly as gemm() plans
 * it (the same kernels, the same K split, the same order of summation), so
 * C equals gemm()'s C bit for bit.  K == 0 gives C = 0.
 *
 * Limit: the scratch gemm() would take for the product -- 4 * M * roundup(K, 32)
 * bytes for a re-strided A, 4 * K * roundup(N, 32) for a re-strided B, and
 * 256 KB per split piece of the K split, each rounded up to 256 bytes -- must
 * not exceed GEMM_NOALLOC_SCRATCH_BYTES (64 MiB).  Aligned products with
 * K, N multiples of 4 need at most the split workspace (14.7 MB at 4096^3,
 * 18.5 MB at 256 x 65536 x 256).  A product that needs more returns
 * GEMM_ERR_SCRATCH_LIMIT and enqueues nothing.
 *
 * Set-up and memory: the first call on a device (that device current) does
 * the library's per-device set-up and looks up the buffer's device address,
 * which loads this part of the library's device code, the 64 MiB buffer
 * with it, onto the device.  Make that first call before the application
 * reserves the rest of the device memory for itself, and before any stream
 * capture; later calls allocate nothing.  With CUDA's lazy module loading
 * (the default) only devices on which this entry point has been called hold
 * the buffer; with CUDA_MODULE_LOADING=EAGER every device on which the
 * process uses this library holds it.  It stays until the process exits.
 *
 * Sharing: every call on a device uses the same buffer, which keeps the last
 * call's contents (nothing in it needs to start at zero: every byte a call
 * reads was written earlier in that call).  Calls whose kernels overlap on
 * the GPU -- on different streams, or from different threads -- race on the
 * buffer and give wrong results: order them on one stream, or synchronise
 * between them.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (64ll * 1024 * 1024)

GEMM_API int gemm_tf32_noalloc(const float* A, const float* B, float* C, int64_t M, int64_t K,
                               int64_t N, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBGEMM_GEMM_H */
