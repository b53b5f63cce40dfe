// ffma_small.cu -- exact binary32 GEMM for small products (mode GEMM_FP32).
//
// The same result as ffma_sgemm.cu: every C_ij is one chain of fused
// multiply-adds with k ascending, C_ij = sum_k A_ik B_kj ("Shared Memory
// Tiling for Matrix Multiplication", opening formula), row-major.  That kernel
// covers C with 128 x 128 tiles, so a small output (128^3 is one tile) runs on
// a handful of SMs, or needs a K split and a second launch to add the pieces.
// This kernel covers C with 32 x 32 tiles, one 64-thread CTA each, 4 x 4
// outputs per thread (the register block of "From 306 ms to 86 ms"), so a
// small product spreads over many SMs in a single launch: 384^2 outputs are
// 144 CTAs.  K is walked in slabs of 16 through a four-slot cp.async ring
// (three slabs in flight: with one CTA per SM there is little else to hide
// the load latency behind; two slots were 25-35 % slower); the
// A slab is stored [k][m] (padded) so that a thread's four rows at one k are
// one 16-byte load; out-of-range elements are zero-filled by the copies and
// out-of-range C elements are not stored -- the first page's section 05
// boundary handling.  ffma_small_fits() says which products take it.
#include <cstdlib>
#include <cstring>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace libgemm {
namespace {

constexpr int kSBM = 32, kSBN = 32, kSBK = 16, kSThreads = 64, kSStages = 4;
constexpr int kSLdA = kSBM + 4;   // floats per k-row of the A slab ([k][m], padded)

// One CTA: the 32 x 32 tile `blockIdx.x` of C, all of K.  Thread t owns rows
// m0 + 4 (t / 8) .. +3 and columns n0 + 4 (t % 8) .. +3.
template <bool kBVec, bool kCVec>
__global__ void __launch_bounds__(kSThreads)
    ffma_small_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K, int tiles_n,
                      const Epilogue epi) {
    __shared__ __align__(16) float sA[kSStages][kSBK][kSLdA];
    __shared__ __align__(16) float sB[kSStages][kSBK][kSBN];
    const int m0 = (int)(blockIdx.x / tiles_n) * kSBM, n0 = (int)(blockIdx.x % tiles_n) * kSBN;
    const int tid = threadIdx.x;
    const int tm = tid / 8, tn = tid % 8;
    const int nkt = (K + kSBK - 1) / kSBK;

    // A: thread t copies row m0 + t % 32, k offsets 8 (t / 32) .. +7 of each
    // slab (a warp's 32 stores at one k land in 32 banks: 36 k + m).
    const int ar = tid % 32, ak = (tid / 32) * 8;
    const bool a_row_ok = m0 + ar < M;
    const float* a_src = a_row_ok ? A + (int64_t)(m0 + ar) * K : A;
    auto load = [&](int kt, int slot) {
        const int k0 = kt * kSBK;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = k0 + ak + j;
            bool ok = a_row_ok && k < K;
            const float* src = ok ? a_src + k : A;
            if (ok) ok = GEMM_DBG_OK(src, A, (int64_t)M * K * 4, 4);
            cp_async_4(smem_u32(&sA[slot][ak + j][ar]), src, ok);
        }
        if constexpr (kBVec) {   // N % 4 == 0 and B 16-byte aligned: 16-byte copies
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int kr = tid / 8 + 8 * r, c = n0 + 4 * (tid % 8);
                bool ok = k0 + kr < K && c < N;
                const float* src = ok ? B + (int64_t)(k0 + kr) * N + c : B;
                if (ok) ok = GEMM_DBG_OK(src, B, (int64_t)K * N * 4, 16);
                cp_async_16(smem_u32(&sB[slot][kr][4 * (tid % 8)]), src, ok);
            }
        } else {
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int kr = tid / 32 + 2 * r, c = n0 + tid % 32;
                bool ok = k0 + kr < K && c < N;
                const float* src = ok ? B + (int64_t)(k0 + kr) * N + c : B;
                if (ok) ok = GEMM_DBG_OK(src, B, (int64_t)K * N * 4, 4);
                cp_async_4(smem_u32(&sB[slot][kr][tid % 32]), src, ok);
            }
        }
    };

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

#pragma unroll
    for (int s = 0; s < kSStages - 1; ++s) {
        if (s < nkt) load(s, s);
        cp_async_commit();
    }
    for (int kt = 0; kt < nkt; ++kt) {
        const int slot = kt % kSStages;
        // slab kt + S - 1 into the slot slab kt - 1 used, freed by the last barrier
        if (kt + kSStages - 1 < nkt) load(kt + kSStages - 1, (kt + kSStages - 1) % kSStages);
        cp_async_commit();
        cp_async_wait<kSStages - 1>();   // slab kt has landed (this thread's copies) ...
        __syncthreads();      // ... and everyone's
#pragma unroll
        for (int k = 0; k < kSBK; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(&sA[slot][k][4 * tm]);
            const float4 b = *reinterpret_cast<const float4*>(&sB[slot][k][4 * tn]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();      // every thread has read this slot before it is refilled
    }
    cp_async_wait<0>();

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = m0 + 4 * tm + i;
        if (row >= M) continue;
        float* crow = C + (int64_t)row * N;
        const int col = n0 + 4 * tn;
        if (kCVec && col < N) {   // N % 4 == 0: all four columns are in range
            if (!GEMM_DBG_OK(crow + col, C, (int64_t)M * N * 4, 16)) continue;
            *reinterpret_cast<float4*>(crow + col) =
                epilogue_apply4(epi, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]), crow + col);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < N && GEMM_DBG_OK(crow + col + j, C, (int64_t)M * N * 4, 4))
                    crow[col + j] = epilogue_apply(epi, acc[i][j], crow + col + j);
        }
    }
}

}  // namespace

// Small products: at most 384^2 outputs and K <= 512.  Against the 128 x 128
// kernel (which takes a K split and a second launch there) on one GB300, L2
// flushed: 32^3 6.8 vs 10.9 us, 128^3 10.9 vs 18.1, 256^3 12.9 vs 18.1, 384^3
// 17.0 vs 20.1, 128 x 512 x 128 19.1 vs 20.1; at 512^3 (31.4 vs 20.2) and for
// longer K (128 x 1024 x 128: 31.4 vs ~21) the 128 x 128 kernel and its split
// win.
bool ffma_small_fits(int64_t M, int64_t N, int64_t K, int num_sms) {
    (void)num_sms;
    // GEMM_FORCE_CONFIG=ffma_small / ffma_tiles128: one kernel for every FP32
    // product (read once per process)
    static const int force = [] {
        const char* f = std::getenv("GEMM_FORCE_CONFIG");
        if (f && std::strcmp(f, "ffma_small") == 0) return 1;
        if (f && std::strcmp(f, "ffma_tiles128") == 0) return -1;
        return 0;
    }();
    if (M <= 0 || N <= 0 || K <= 0 || force < 0) return false;
    return force > 0 || (M * N <= kSmallMaxMN && K <= kSmallMaxK);
}

cudaError_t launch_ffma_small(const float* A, const float* B, float* C, int M, int N, int K,
                              bool b_vec, bool c_vec, const Epilogue& epi, cudaStream_t stream) {
    const int64_t tiles_m = (M + kSBM - 1) / kSBM, tiles_n = (N + kSBN - 1) / kSBN;
    const int64_t tiles = tiles_m * tiles_n;
    if (tiles <= 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)tiles), block(kSThreads);
    const int tn = (int)tiles_n;
    if (b_vec && c_vec)
        ffma_small_kernel<true, true><<<grid, block, 0, stream>>>(A, B, C, M, N, K, tn, epi);
    else if (b_vec)
        ffma_small_kernel<true, false><<<grid, block, 0, stream>>>(A, B, C, M, N, K, tn, epi);
    else if (c_vec)
        ffma_small_kernel<false, true><<<grid, block, 0, stream>>>(A, B, C, M, N, K, tn, epi);
    else
        ffma_small_kernel<false, false><<<grid, block, 0, stream>>>(A, B, C, M, N, K, tn, epi);
    return cudaGetLastError();
}

LIBGEMM_DEBUG_READER(ffma_small_debug_flags)

}  // namespace libgemm
