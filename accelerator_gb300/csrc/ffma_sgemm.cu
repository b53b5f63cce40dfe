// ffma_sgemm.cu -- exact binary32 GEMM on the CUDA cores (mode GEMM_FP32).
//
// C_ij = sum_k A_ik B_kj ("Shared Memory Tiling for Matrix Multiplication",
// opening formula), row-major as in "Matrix Multiplication -- Naive to
// Tiled", section 02.  Every C_ij is one chain of fused multiply-adds with k
// ascending, so the result is the sequential binary32 sum of exact products.
//
// Design (GB300 rather than the pages' 16x16/32x32 tiles):
//   * A CTA of 256 threads owns a 128 x 128 tile of C; a thread owns an 8 x 8
//     register block, laid out as 2 x 2 sub-blocks of 4 x 4 so each fragment
//     is one 128-bit shared-memory load.  Per k a thread does 64 FMAs for 4
//     fragment loads -- the register blocking of "From 306 ms to 86 ms"
//     (4 x 4 there) and "Further Optimisation Ideas" of the first page,
//     taken to 8 x 8.
//   * K is walked in slabs of 16 through a 4-stage ring of shared-memory
//     buffers filled by cp.async, so global loads of later slabs overlap the
//     arithmetic on the current one (the page's "double buffering", deeper).
//   * The A slab is stored transposed (k-major, [k][m], padded by 4 floats) so
//     that a thread's 4 consecutive rows of A at one k are one 128-bit load;
//     the element-wise cp.async that does the transposition is arranged so a
//     warp's 32 stores hit 32 different banks.  B slabs are copied 16 bytes
//     at a time when rows are 16-byte aligned, else 4 bytes at a time.
//   * Out-of-range elements of the last slabs are zero-filled by the copy
//     (source size 0) and out-of-range C elements are never stored -- the
//     boundary handling of the first page's section 05, for any M, K, N.
//   * Tiles are visited in groups of 8 tile-rows so CTAs running together
//     share A and B slabs in L2.
#include "kernels.h"
#include "ptx.cuh"

namespace libgemm {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16;
constexpr int kWM = 64, kWN = 32;               // warp tile
constexpr int kStages = 4;
constexpr int kThreads = (kBM / kWM) * (kBN / kWN) * 32;  // 256
constexpr int kLM = kWM / 8, kLN = kWN / 8;     // lanes along m / n: 8 x 4
constexpr int kPadA = 4;
constexpr int kLdA = kBM + kPadA;               // floats per k-row of the A slab
constexpr int kLdB = kBN;
constexpr int kAStage = kBK * kLdA;             // floats
constexpr int kBStage = kBK * kLdB;
constexpr size_t kSmemBytes = size_t(kStages) * (kAStage + kBStage) * sizeof(float);
constexpr int kGroupM = 8;

static_assert(kLM * kLN == 32, "a warp is 32 lanes");
static_assert(kThreads == 256, "launch shape");
static_assert((kBM * kBK) % kThreads == 0 && (kBK * kBN) % (4 * kThreads) == 0, "load split");

// Issue the copies of K-slab `kt` into ring slot `slot`.
template <bool kBVec>
__device__ __forceinline__ void load_slab(const float* __restrict__ A, const float* __restrict__ B,
                                          float* sA, float* sB, int M, int N, int K, int m0,
                                          int n0, int kt, int tid) {
    const int k0 = kt * kBK;
    // A: 128 x 16 elements, 8 per thread.  A pass covers 8 consecutive k of
    // 32 rows; lanes 0-7 take one row, so a warp reads 4 x 32 contiguous bytes
    // and its transposed stores land in banks (4*k + row) mod 32, all distinct.
    constexpr int kRowsPerPass = kThreads / 8;            // 32
    constexpr int kPassesPerK8 = kBM / kRowsPerPass;      // 4
#pragma unroll
    for (int r = 0; r < (kBM * kBK) / kThreads; ++r) {
        const int kk = (tid & 7) + 8 * (r / kPassesPerK8);
        const int mm = (tid >> 3) + kRowsPerPass * (r % kPassesPerK8);
        const int gm = m0 + mm, gk = k0 + kk;
        const bool ok = gm < M && gk < K;
        const float* src = ok ? A + (int64_t)gm * K + gk : A;
        cp_async_4(smem_u32(sA + kk * kLdA + mm), src, ok);
    }
    if constexpr (kBVec) {
        // B: 16 rows x 32 chunks of 16 bytes, 2 chunks per thread; a warp copies
        // one contiguous 512-byte row piece.
#pragma unroll
        for (int r = 0; r < (kBK * kBN) / (4 * kThreads); ++r) {
            const int c = r * kThreads + tid;
            const int kk = c / (kBN / 4), nn = (c % (kBN / 4)) * 4;
            const int gk = k0 + kk, gn = n0 + nn;
            const bool ok = gk < K && gn < N;   // N % 4 == 0: the chunk is all in or all out
            const float* src = ok ? B + (int64_t)gk * N + gn : B;
            cp_async_16(smem_u32(sB + kk * kLdB + nn), src, ok);
        }
    } else {
#pragma unroll
        for (int r = 0; r < (kBK * kBN) / kThreads; ++r) {
            const int e = r * kThreads + tid;
            const int kk = e / kBN, nn = e % kBN;
            const int gk = k0 + kk, gn = n0 + nn;
            const bool ok = gk < K && gn < N;
            const float* src = ok ? B + (int64_t)gk * N + gn : B;
            cp_async_4(smem_u32(sB + kk * kLdB + nn), src, ok);
        }
    }
}

template <bool kBVec, bool kCVec>
__global__ void __launch_bounds__(kThreads, 1)
    ffma_sgemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K, int tiles_m, int tiles_n) {
    extern __shared__ __align__(16) float smem[];
    float* sA = smem;                          // kStages x [kBK][kLdA]
    float* sB = smem + kStages * kAStage;      // kStages x [kBK][kLdB]

    // Grouped raster: consecutive CTAs walk down a group of kGroupM tile-rows.
    const int tile = blockIdx.x;
    const int per_group = kGroupM * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * kGroupM;
    const int gsize = min(tiles_m - first_m, kGroupM);
    const int tm = first_m + (tile % per_group) % gsize;
    const int tn = (tile % per_group) / gsize;
    const int m0 = tm * kBM, n0 = tn * kBN;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm0 = (warp / (kBN / kWN)) * kWM;
    const int wn0 = (warp % (kBN / kWN)) * kWN;
    const int lm = lane % kLM, ln = lane / kLM;
    const int am = wm0 + lm * 4;               // rows am..am+3 and am+kWM/2..+3
    const int bn = wn0 + ln * 4;               // cols bn..bn+3 and bn+kWN/2..+3

    const int nkt = (K + kBK - 1) / kBK;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nkt)
            load_slab<kBVec>(A, B, sA + s * kAStage, sB + s * kBStage, M, N, K, m0, n0, s, tid);
        cp_async_commit();
    }

    for (int kt = 0; kt < nkt; ++kt) {
        cp_async_wait<kStages - 2>();   // slab kt has landed (this thread's copies)
        __syncthreads();                // ... everyone's; and slot (kt-1) is free
        {
            const int nxt = kt + kStages - 1;
            if (nxt < nkt) {
                const int slot = nxt % kStages;
                load_slab<kBVec>(A, B, sA + slot * kAStage, sB + slot * kBStage, M, N, K, m0, n0,
                                 nxt, tid);
            }
            cp_async_commit();
        }
        const float* a_s = sA + (kt % kStages) * kAStage;
        const float* b_s = sB + (kt % kStages) * kBStage;
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(a_s + k * kLdA + am);
            const float4 a1 = *reinterpret_cast<const float4*>(a_s + k * kLdA + am + kWM / 2);
            const float4 b0 = *reinterpret_cast<const float4*>(b_s + k * kLdB + bn);
            const float4 b1 = *reinterpret_cast<const float4*>(b_s + k * kLdB + bn + kWN / 2);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // Store the 8 x 8 block: guarded against M and N.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + am + (i < 4 ? i : kWM / 2 + (i - 4));
        if (row >= M) continue;
        float* crow = C + (int64_t)row * N;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + bn + h * (kWN / 2);
            if (kCVec && col < N) {   // N % 4 == 0: all four columns are in range
                *reinterpret_cast<float4*>(crow + col) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < N) crow[col + j] = acc[i][4 * h + j];
            }
        }
    }
}

template <bool BV, bool CV>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(ffma_sgemm_kernel<BV, CV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

}  // namespace

cudaError_t ffma_setup() {
    cudaError_t e;
    if ((e = set_smem_attr<false, false>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<true, false>()) != cudaSuccess) return e;
    return set_smem_attr<true, true>();
}

cudaError_t launch_ffma_sgemm(const float* A, const float* B, float* C, int M, int N, int K,
                              bool b_vec, bool c_vec, cudaStream_t stream) {
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = (int64_t)tiles_m * tiles_n;
    if (tiles <= 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dim3 grid((unsigned)tiles), block(kThreads);
    if (b_vec && c_vec)
        ffma_sgemm_kernel<true, true><<<grid, block, kSmemBytes, stream>>>(A, B, C, M, N, K, tiles_m, tiles_n);
    else if (b_vec)
        ffma_sgemm_kernel<true, false><<<grid, block, kSmemBytes, stream>>>(A, B, C, M, N, K, tiles_m, tiles_n);
    else if (c_vec)
        ffma_sgemm_kernel<false, true><<<grid, block, kSmemBytes, stream>>>(A, B, C, M, N, K, tiles_m, tiles_n);
    else
        ffma_sgemm_kernel<false, false><<<grid, block, kSmemBytes, stream>>>(A, B, C, M, N, K, tiles_m, tiles_n);
    return cudaGetLastError();
}

}  // namespace libgemm
