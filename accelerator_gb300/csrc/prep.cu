// prep.cu -- small helper kernels of libgemm.
//
//   restride    copies an operand into a buffer whose row stride is a multiple
//               of 16 bytes, for the tensor-core path when TMA cannot describe
//               the caller's layout (e.g. K = 777 floats: 3108-byte rows).
//   to_bf16 / to_tf32  the rounding passes of GEMM_FP32_VIA_BF16 and
//               GEMM_TF32_RN (to nearest; ties to even / away from zero).
//   fill_zero   C := 0 for K == 0 (the empty sum).
//   scale       C := beta * C, the generalised product when alpha == 0 or K == 0.
//   splitk_reduce  adds the K-split partials of the tensor kernel in split
//               order and applies the epilogue.
//   wait_selftest  one CTA waits on an mbarrier that nothing completes, to
//               show the bounded wait gives up and reports instead of hanging.
#include <cuda_bf16.h>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace libgemm {
namespace {

// Rows of row_bytes bytes from stride src_ld to stride dst_ld (both in
// bytes), copied V bytes at a time -- V the widest unit that divides both
// bases and both strides -- and the rows' last row_bytes % V bytes two at a
// time (elements are 2 or 4 bytes); the padding after each destination row
// is zeroed.  One flat index runs over all (row, unit) pairs, so
// consecutive threads copy consecutive units and every thread has several
// independent copies in flight.
template <typename V>
__global__ void restride_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                int64_t rows, int64_t row_bytes, int64_t src_ld, int64_t dst_ld) {
    const int64_t nvec = row_bytes / (int64_t)sizeof(V), tail0 = nvec * (int64_t)sizeof(V);
    const int64_t ntail = (row_bytes - tail0) / 2;
    [[maybe_unused]] const int64_t src_bytes = (rows - 1) * src_ld + row_bytes;
    [[maybe_unused]] const int64_t dst_bytes = rows * dst_ld;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
#pragma unroll 4
    for (int64_t u = first; u < rows * nvec; u += step) {
        const int64_t r = u / nvec, c = u - r * nvec;
        const V* sp = reinterpret_cast<const V*>(src + r * src_ld) + c;
        V* dp = reinterpret_cast<V*>(dst + r * dst_ld) + c;
        if (GEMM_DBG_OK(sp, src, src_bytes, sizeof(V)) && GEMM_DBG_OK(dp, dst, dst_bytes, sizeof(V)))
            *dp = *sp;
    }
    for (int64_t u = first; u < rows * ntail; u += step) {
        const int64_t r = u / ntail, b = tail0 + 2 * (u - r * ntail);
        const uint16_t* sp = reinterpret_cast<const uint16_t*>(src + r * src_ld + b);
        uint16_t* dp = reinterpret_cast<uint16_t*>(dst + r * dst_ld + b);
        if (GEMM_DBG_OK(sp, src, src_bytes, 2) && GEMM_DBG_OK(dp, dst, dst_bytes, 2)) *dp = *sp;
    }
    // each destination row's padding (row_bytes .. dst_ld) is zeroed: a
    // reader may load it with the row's last vector
    const int64_t npad = (dst_ld - row_bytes) / 2;
    for (int64_t u = first; u < rows * npad; u += step) {
        const int64_t r = u / npad, b = row_bytes + 2 * (u - r * npad);
        uint16_t* dp = reinterpret_cast<uint16_t*>(dst + r * dst_ld + b);
        if (GEMM_DBG_OK(dp, dst, dst_bytes, 2)) *dp = 0;
    }
}

// float -> bfloat16, round to nearest even, into rows of stride dst_ld.  The
// vector form reads 4 floats (16 bytes) and writes 4 bf16 (8 bytes) per step;
// it needs cols % 4 == 0, 16-byte aligned src and 8-byte aligned dst rows.
__global__ void to_bf16_v4_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                  int64_t rows, int64_t cols4, int64_t dst_ld4) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cols4;
             c += (int64_t)gridDim.x * blockDim.x) {
            if (!GEMM_DBG_OK(src + r * cols4 + c, src, rows * cols4 * 16, 16) ||
                !GEMM_DBG_OK(dst + r * dst_ld4 + c, dst, rows * dst_ld4 * 8, 8))
                continue;
            const float4 v = src[r * cols4 + c];
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
            dst[r * dst_ld4 + c] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                              *reinterpret_cast<const uint32_t*>(&hi));
        }
}

// Both operands in one launch: rows [0, rows_a) of the combined index are
// A's, the rest B's.  A block converts one row at a time, each thread four
// 16-byte chunks per pass with all four loads issued before any store, so
// about 64 bytes per thread are in flight (one chunk per thread leaves the
// loads too few to cover HBM latency).  Needs the vector form's alignment.
struct Bf16Job {
    const float4* src;
    uint2* dst;
    int64_t rows, cols4, dst_ld4;
};

// float -> TF32, round to nearest with ties away from zero (cvt.rna.tf32.f32),
// kept as a binary32 whose 13 low fraction bits are zero.
__device__ __forceinline__ float round_tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r & 0xFFFFE000u);
}

// The TF32 rounding pass of GEMM_TF32_RN: both operands in one launch, laid
// out like the bfloat16 pass (one row per block and pass, four 16-byte
// loads in flight per thread), writing rounded floats into rows of stride
// dst_ld4 float4s.
struct Tf32Job {
    const float4* src;
    float4* dst;
    int64_t rows, cols4, dst_ld4;
};

__global__ void __launch_bounds__(256) to_tf32_pair_kernel(Tf32Job a, Tf32Job b) {
    grid_launch_dependents();   // the MMA kernel may start its set-up meanwhile
    const int64_t total = a.rows + b.rows;
    for (int64_t rr = blockIdx.x; rr < total; rr += gridDim.x) {
        const bool in_a = rr < a.rows;
        const Tf32Job& j = in_a ? a : b;
        const int64_t r = in_a ? rr : rr - a.rows;
        const float4* s = j.src + r * j.cols4;
        float4* d = j.dst + r * j.dst_ld4;
        for (int64_t c0 = threadIdx.x; c0 < j.cols4; c0 += 4 * (int64_t)blockDim.x) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t c = c0 + q * (int64_t)blockDim.x;
                v[q] = c < j.cols4 && GEMM_DBG_OK(s + c, j.src, j.rows * j.cols4 * 16, 16)
                           ? __ldcs(s + c)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t c = c0 + q * (int64_t)blockDim.x;
                if (c < j.cols4 && GEMM_DBG_OK(d + c, j.dst, j.rows * j.dst_ld4 * 16, 16))
                    d[c] = make_float4(round_tf32_rna(v[q].x), round_tf32_rna(v[q].y),
                                       round_tf32_rna(v[q].z), round_tf32_rna(v[q].w));
            }
        }
    }
}

// Element-wise form for rows that are not whole 16-byte chunks.
__global__ void to_tf32_kernel(const float* __restrict__ src, float* __restrict__ dst,
                               int64_t rows, int64_t cols, int64_t dst_ld) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cols;
             c += (int64_t)gridDim.x * blockDim.x)
            if (GEMM_DBG_OK(src + r * cols + c, src, rows * cols * 4, 4) &&
                GEMM_DBG_OK(dst + r * dst_ld + c, dst, rows * dst_ld * 4, 4))
                dst[r * dst_ld + c] = round_tf32_rna(src[r * cols + c]);
}

__global__ void __launch_bounds__(256) to_bf16_pair_kernel(Bf16Job a, Bf16Job b) {
    grid_launch_dependents();   // the MMA kernel may start its set-up meanwhile
    const int64_t total = a.rows + b.rows;
    for (int64_t rr = blockIdx.x; rr < total; rr += gridDim.x) {
        const bool in_a = rr < a.rows;
        const Bf16Job& j = in_a ? a : b;
        const int64_t r = in_a ? rr : rr - a.rows;
        const float4* s = j.src + r * j.cols4;
        uint2* d = j.dst + r * j.dst_ld4;
        for (int64_t c0 = threadIdx.x; c0 < j.cols4; c0 += 4 * (int64_t)blockDim.x) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t c = c0 + q * (int64_t)blockDim.x;
                v[q] = c < j.cols4 && GEMM_DBG_OK(s + c, j.src, j.rows * j.cols4 * 16, 16)
                           ? __ldcs(s + c)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t c = c0 + q * (int64_t)blockDim.x;
                if (c < j.cols4 && GEMM_DBG_OK(d + c, j.dst, j.rows * j.dst_ld4 * 8, 8)) {
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[q].x, v[q].y);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[q].z, v[q].w);
                    d[c] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                      *reinterpret_cast<const uint32_t*>(&hi));
                }
            }
        }
    }
}

__global__ void to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                               int64_t rows, int64_t cols, int64_t dst_ld) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < cols;
             c += (int64_t)gridDim.x * blockDim.x)
            if (GEMM_DBG_OK(src + r * cols + c, src, rows * cols * 4, 4) &&
                GEMM_DBG_OK(dst + r * dst_ld + c, dst, rows * dst_ld * 2, 2))
                dst[r * dst_ld + c] = __float2bfloat16_rn(src[r * cols + c]);
}

__global__ void fill_zero_kernel(float* __restrict__ C, int64_t n) {
    // a kernel launched after this one with programmatic stream serialisation
    // (the FFMA stream-K kernel) may start at once; it waits for the zeros
    // before it reads them
    grid_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        if (GEMM_DBG_OK(C + i, C, n * 4, 4)) C[i] = 0.0f;
}

// C := beta * C, one rounding per element (alpha == 0 or K == 0 with beta != 0).
__global__ void scale_kernel(float* __restrict__ C, int64_t n, float beta) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        if (GEMM_DBG_OK(C + i, C, n * 4, 4)) C[i] = __fmul_rn(beta, C[i]);
}

// K-split fix-up: C_ij := epilogue(p_0 + p_1 + ... + p_{S-1}), the partials
// p_s = ws[(s * ws_rows + i) * ws_ld + j] added in split order (the same sum
// on every run).  Each thread loads four partials before adding them, so
// several loads are in flight.  Vector form: four columns per thread, for
// N % 4 == 0 and 16-byte aligned rows of C and of ws.
template <bool kVec>
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, int splits, int64_t ws_rows,
                         int64_t ws_ld, float* __restrict__ C, int64_t M, int64_t N,
                         const Epilogue epi) {
    constexpr int W = kVec ? 4 : 1;
    const int64_t nw = (N + W - 1) / W, units = M * nw;
    const int64_t sstride = ws_rows * ws_ld;
    grid_dependency_wait();   // the partials' kernel is complete and its writes visible
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = u / nw, j = (u - i * nw) * W;
        const float* p = ws + i * ws_ld + j;
        if (!GEMM_DBG_OK(p, ws, splits * sstride * 4, 4 * W) ||
            !GEMM_DBG_OK(p + (splits - 1) * sstride, ws, splits * sstride * 4, 4 * W) ||
            !GEMM_DBG_OK(C + i * N + j, C, M * N * 4, 4 * W))
            continue;
        if constexpr (kVec) {
            float4 acc = __ldcg(reinterpret_cast<const float4*>(p));
            int s = 1;
            for (; s + 4 <= splits; s += 4) {
                float4 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    v[q] = __ldcg(reinterpret_cast<const float4*>(p + (s + q) * sstride));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc.x += v[q].x, acc.y += v[q].y, acc.z += v[q].z, acc.w += v[q].w;
            }
            for (; s < splits; ++s) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(p + s * sstride));
                acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
            }
            float* c = C + i * N + j;
            *reinterpret_cast<float4*>(c) = epilogue_apply4(epi, acc, c);
        } else {
            float acc = __ldcg(p);
            int s = 1;
            for (; s + 4 <= splits; s += 4) {
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = __ldcg(p + (s + q) * sstride);
#pragma unroll
                for (int q = 0; q < 4; ++q) acc += v[q];
            }
            for (; s < splits; ++s) acc += __ldcg(p + s * sstride);
            float* c = C + i * N + j;
            *c = epilogue_apply(epi, acc, c);
        }
    }
}

__global__ void wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // No thread and no copy ever arrives: phase 0 never completes.
        (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_restride(const void* src, void* dst, int64_t rows, int64_t cols,
                            int64_t src_ld, int64_t dst_ld, int es, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (es != 2 && es != 4) return cudaErrorInvalidValue;
    const int64_t row_bytes = cols * es, sld = src_ld * es, dld = dst_ld * es;
    const uint64_t align = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                           (uint64_t)sld | (uint64_t)dld;
    const int v = (align & 15u) == 0 ? 16 : (align & 7u) == 0 ? 8 : (align & 3u) == 0 ? 4 : 2;
    // up to 16 blocks of 256 threads an SM, each thread a few units
    const int threads = 256;
    const int64_t units = rows * (row_bytes / v) + rows * ((row_bytes % v) / 2);
    int64_t blocks = (units + threads - 1) / threads;
    blocks = blocks < 1 ? 1 : (blocks > 152 * 16 ? 152 * 16 : blocks);
    const dim3 grid((unsigned)blocks);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    uint8_t* d = static_cast<uint8_t*>(dst);
    if (v == 16)
        restride_kernel<uint4><<<grid, threads, 0, stream>>>(s, d, rows, row_bytes, sld, dld);
    else if (v == 8)
        restride_kernel<uint2><<<grid, threads, 0, stream>>>(s, d, rows, row_bytes, sld, dld);
    else if (v == 4)
        restride_kernel<uint32_t><<<grid, threads, 0, stream>>>(s, d, rows, row_bytes, sld, dld);
    else
        restride_kernel<uint16_t><<<grid, threads, 0, stream>>>(s, d, rows, row_bytes, sld, dld);
    return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float* src, void* dst, int64_t rows, int64_t cols,
                           int64_t dst_ld, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int threads = 256;
    const unsigned gy = (unsigned)(rows < 65535 ? rows : 65535);
    if (cols % 4 == 0 && dst_ld % 4 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
        const int64_t c4 = cols / 4, bx = (c4 + threads - 1) / threads;
        dim3 grid((unsigned)(bx < 16 ? bx : 16), gy);
        to_bf16_v4_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                        static_cast<uint2*>(dst), rows, c4, dst_ld / 4);
    } else {
        const int64_t bx = (cols + threads - 1) / threads;
        dim3 grid((unsigned)(bx < 64 ? bx : 64), gy);
        to_bf16_kernel<<<grid, threads, 0, stream>>>(src, static_cast<__nv_bfloat16*>(dst), rows,
                                                     cols, dst_ld);
    }
    return cudaGetLastError();
}

cudaError_t launch_to_bf16_pair(const float* a, void* a_dst, int64_t a_rows, int64_t a_cols,
                                int64_t a_ld, const float* b, void* b_dst, int64_t b_rows,
                                int64_t b_cols, int64_t b_ld, cudaStream_t stream, int* launches) {
    auto vec_ok = [](const float* src, const void* dst, int64_t cols, int64_t ld) {
        return cols % 4 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
               (reinterpret_cast<uintptr_t>(dst) & 7u) == 0;
    };
    *launches = 0;
    if (a_rows <= 0 || a_cols <= 0 || b_rows <= 0 || b_cols <= 0 ||
        !vec_ok(a, a_dst, a_cols, a_ld) || !vec_ok(b, b_dst, b_cols, b_ld)) {
        cudaError_t e = launch_to_bf16(a, a_dst, a_rows, a_cols, a_ld, stream);
        ++*launches;
        if (e == cudaSuccess) {
            e = launch_to_bf16(b, b_dst, b_rows, b_cols, b_ld, stream);
            ++*launches;
        }
        return e;
    }
    const Bf16Job ja{reinterpret_cast<const float4*>(a), static_cast<uint2*>(a_dst), a_rows,
                     a_cols / 4, a_ld / 4};
    const Bf16Job jb{reinterpret_cast<const float4*>(b), static_cast<uint2*>(b_dst), b_rows,
                     b_cols / 4, b_ld / 4};
    const int64_t rows = a_rows + b_rows;
    const unsigned grid = (unsigned)(rows < (1 << 20) ? rows : (1 << 20));
    to_bf16_pair_kernel<<<grid, 256, 0, stream>>>(ja, jb);
    *launches = 1;
    return cudaGetLastError();
}

cudaError_t launch_to_tf32_pair(const float* a, float* a_dst, int64_t a_rows, int64_t a_cols,
                                int64_t a_ld, const float* b, float* b_dst, int64_t b_rows,
                                int64_t b_cols, int64_t b_ld, cudaStream_t stream, int* launches) {
    auto vec_ok = [](const float* src, const float* dst, int64_t cols, int64_t ld) {
        return cols % 4 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
               (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    };
    *launches = 0;
    if (a_rows <= 0 || a_cols <= 0 || b_rows <= 0 || b_cols <= 0 ||
        !vec_ok(a, a_dst, a_cols, a_ld) || !vec_ok(b, b_dst, b_cols, b_ld)) {
        const float* src[2] = {a, b};
        float* dst[2] = {a_dst, b_dst};
        const int64_t rows[2] = {a_rows, b_rows}, cols[2] = {a_cols, b_cols}, ld[2] = {a_ld, b_ld};
        for (int t = 0; t < 2; ++t) {
            if (rows[t] <= 0 || cols[t] <= 0) continue;
            const int64_t bx = (cols[t] + 255) / 256;
            dim3 grid((unsigned)(bx < 64 ? bx : 64), (unsigned)(rows[t] < 65535 ? rows[t] : 65535));
            to_tf32_kernel<<<grid, 256, 0, stream>>>(src[t], dst[t], rows[t], cols[t], ld[t]);
            ++*launches;
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    const Tf32Job ja{reinterpret_cast<const float4*>(a), reinterpret_cast<float4*>(a_dst), a_rows,
                     a_cols / 4, a_ld / 4};
    const Tf32Job jb{reinterpret_cast<const float4*>(b), reinterpret_cast<float4*>(b_dst), b_rows,
                     b_cols / 4, b_ld / 4};
    const int64_t rows = a_rows + b_rows;
    const unsigned grid = (unsigned)(rows < (1 << 20) ? rows : (1 << 20));
    to_tf32_pair_kernel<<<grid, 256, 0, stream>>>(ja, jb);
    *launches = 1;
    return cudaGetLastError();
}

cudaError_t launch_fill_zero(float* C, int64_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    fill_zero_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(C, n);
    return cudaGetLastError();
}

cudaError_t launch_scale(float* C, int64_t n, float beta, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    scale_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(C, n, beta);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t ws_rows, int64_t ws_ld,
                                 float* C, int64_t M, int64_t N, bool c_vec, const Epilogue& epi,
                                 int num_sms, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (splits < 1 || ws_rows < M || ws_ld < N) return cudaErrorInvalidValue;
    const bool vec = c_vec && N % 4 == 0 && ws_ld % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(ws) & 15u) == 0;
    const int64_t units = M * (vec ? N / 4 : N);
    const int64_t blocks = (units + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 16;   // two rounds of 8 resident 256-thread blocks
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = kUsePdl ? 1 : 0;
    const cudaError_t e =
        vec ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<true>, ws, splits, ws_rows, ws_ld, C, M,
                                 N, epi)
            : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<false>, ws, splits, ws_rows, ws_ld, C,
                                 M, N, epi);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

LIBGEMM_DEBUG_READER(prep_debug_flags)

}  // namespace libgemm
