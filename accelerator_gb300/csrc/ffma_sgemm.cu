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
constexpr int kMinBlocks = 2;                   // CTAs per SM the register budget allows
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

// The copies of one thread, planned once per tile so that issuing the copies
// of a K slab is a few pointer and address additions.  Slabs that lie wholly
// inside K need no K check; only the last one, when K % kBK != 0, has it.
//
// A: kBM x kBK elements, kAPer per thread.  A pass covers 8 consecutive k of
// kThreads/8 rows; lanes 0-7 take one row, so a warp reads 4 x 32 contiguous
// bytes and its transposed stores land in banks (4*k + row) mod 32, all
// distinct.  B: rows of kBN columns copied 16 bytes (kBVec) or 4 bytes per
// copy, a warp covering one contiguous 512- or 128-byte row piece.
template <bool kBVec>
struct SlabLoader {
    static constexpr int kRowsPerPass = kThreads / 8;              // 32 rows of A per pass
    static constexpr int kARowGroups = kBM / kRowsPerPass;         // 4
    static constexpr int kAPer = (kBM * kBK) / kThreads;           // 8 copies of A
    static constexpr int kBElems = kBVec ? 4 : 1;                  // floats per B copy
    static constexpr int kBPerRow = kBN / kBElems;                 // copies per B row
    static constexpr int kBRowsPerPass = kThreads / kBPerRow;      // 8 (vec) or 2
    static constexpr int kBPer = kBK / kBRowsPerPass;              // 2 (vec) or 8
    static_assert(kThreads % kBPerRow == 0 && kBK % kBRowsPerPass == 0, "B split");

    const float* a_base;               // A itself: source of zero-size copies
    const float* a_ptr;                // &A[m0 + tid/8][tid % 8]
    const float* b_ptr;                // &B[tid / kBPerRow][n0 + column of this thread]
    int64_t a_group_step;              // kRowsPerPass * K: to the next row group of A
    int64_t n;                         // N, the row stride of B
    uint32_t a_row_ok;                 // bit j: row of a_row[j] < M
    bool b_col_ok;
    int a_k, b_k;                      // this thread's k offset within a slab (A, B)
    uint32_t a_dst, b_dst;             // shared addresses in ring slot 0

    __device__ __forceinline__ SlabLoader(const float* A, const float* B, float* sA, float* sB,
                                          int M, int N, int K, int m0, int n0, int tid) {
        const int ar = tid >> 3;
        a_k = tid & 7;
        a_base = A;
        a_row_ok = 0;
#pragma unroll
        for (int j = 0; j < kARowGroups; ++j)
            a_row_ok |= (m0 + ar + kRowsPerPass * j < M ? 1u : 0u) << j;
        a_ptr = A + (int64_t)(m0 + ar) * K + a_k;   // only dereferenced for rows < M
        a_group_step = (int64_t)kRowsPerPass * K;
        a_dst = smem_u32(sA + a_k * kLdA + ar);
        b_k = tid / kBPerRow;
        const int bc = (tid % kBPerRow) * kBElems;
        b_col_ok = n0 + bc < N;   // vec: N % 4 == 0, so the whole chunk is in or out
        b_ptr = b_col_ok ? B + (int64_t)b_k * N + n0 + bc : B;
        n = N;
        b_dst = smem_u32(sB + b_k * kLdB + bc);
    }

    // Copies of slab kt into ring slot `slot` for a tile wholly inside M and N
    // and a slab wholly inside K: no checks, and every copy of a row group is
    // one base pointer plus a constant offset.
    __device__ __forceinline__ void load_interior(int kt, int slot) const {
        const int k0 = kt * kBK;
        const uint32_t adst = a_dst + (uint32_t)(slot * kAStage * 4);
#pragma unroll
        for (int j = 0; j < kARowGroups; ++j) {
            const float* row = a_ptr + j * a_group_step + k0;
#pragma unroll
            for (int g = 0; g < kAPer / kARowGroups; ++g)
                cp_async_4(adst + (uint32_t)((8 * g * kLdA + kRowsPerPass * j) * 4), row + 8 * g);
        }
        const uint32_t bdst = b_dst + (uint32_t)(slot * kBStage * 4);
        const float* bsrc = b_ptr + (int64_t)k0 * n;
#pragma unroll
        for (int r = 0; r < kBPer; ++r) {
            const float* src = bsrc + (int64_t)(kBRowsPerPass * r) * n;
            const uint32_t dst = bdst + (uint32_t)(kBRowsPerPass * r * kLdB * 4);
            if constexpr (kBVec)
                cp_async_16(dst, src);
            else
                cp_async_4(dst, src);
        }
    }

    // Copies of slab kt into ring slot `slot`, each checked against M, N and
    // (check_k, for the last, partial slab) K.
    __device__ __forceinline__ void load(int kt, int slot, int K, bool check_k) const {
        const int k0 = kt * kBK;
        const uint32_t adst = a_dst + (uint32_t)(slot * kAStage * 4);
#pragma unroll
        for (int r = 0; r < kAPer; ++r) {
            const int j = r % kARowGroups, g = r / kARowGroups;   // row group, 8-k group
            const int kk = k0 + 8 * g;
            bool ok = (a_row_ok >> j) & 1u;
            if (check_k) ok = ok && (kk + a_k < K);
            const float* src = ok ? a_ptr + j * a_group_step + kk : a_base;
            cp_async_4(adst + (uint32_t)((8 * g * kLdA + kRowsPerPass * j) * 4), src, ok);
        }
        const uint32_t bdst = b_dst + (uint32_t)(slot * kBStage * 4);
        const float* bsrc = b_ptr + (int64_t)k0 * n;
#pragma unroll
        for (int r = 0; r < kBPer; ++r) {
            bool ok = b_col_ok;
            if (check_k) ok = ok && (k0 + kBRowsPerPass * r + b_k < K);
            const float* src = ok ? bsrc + (int64_t)(kBRowsPerPass * r) * n : b_ptr;
            const uint32_t dst = bdst + (uint32_t)(kBRowsPerPass * r * kLdB * 4);
            if constexpr (kBVec)
                cp_async_16(dst, src, ok);
            else
                cp_async_4(dst, src, ok);
        }
    }
};

// One CTA computes one tile of C over the K slabs [kt_begin, kt_end).  The
// first dp_tiles tiles (in raster order) are computed whole.  Each remaining
// tile is split into `splits` consecutive K ranges computed by different
// CTAs, so that the last, partial wave of tiles still fills the GPU; each
// such CTA writes its partial tile to `partial`, and the last of them to
// finish (an atomic counter per tile) adds the partials in split order and
// stores C.  The sum is then ((p0 + p1) + p2) + ..., the same on every run.
template <bool kBVec, bool kCVec>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    ffma_sgemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K, int tiles_m, int tiles_n,
                      int dp_tiles, int splits, float* __restrict__ partial,
                      unsigned* __restrict__ counters) {
    extern __shared__ __align__(16) float smem[];
    float* sA = smem;                          // kStages x [kBK][kLdA]
    float* sB = smem + kStages * kAStage;      // kStages x [kBK][kLdB]
    __shared__ unsigned s_last;

    const int nkt = (K + kBK - 1) / kBK;
    int tile, part = 0, kt_begin = 0, kt_end = nkt;
    if ((int)blockIdx.x < dp_tiles) {
        tile = blockIdx.x;
    } else {
        const int u = blockIdx.x - dp_tiles;
        tile = dp_tiles + u / splits;
        part = u % splits;
        kt_begin = (int)((int64_t)nkt * part / splits);
        kt_end = (int)((int64_t)nkt * (part + 1) / splits);
    }

    // Grouped raster: consecutive tiles walk down a group of kGroupM tile-rows.
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

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    const SlabLoader<kBVec> loader(A, B, sA, sB, M, N, K, m0, n0, tid);
    const int full_slabs = K / kBK;   // slabs kt < full_slabs lie wholly inside K
    const int nloc = kt_end - kt_begin;

    // Slabs before interior_end can take the unchecked copies.
    const bool interior = m0 + kBM <= M && n0 + kBN <= N;
    const int interior_end = interior ? full_slabs : 0;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nloc) {
            const int kt = kt_begin + s;
            if (kt < interior_end) loader.load_interior(kt, s);
            else loader.load(kt, s, K, kt >= full_slabs);
        }
        cp_async_commit();
    }

    for (int i = 0; i < nloc; ++i) {
        cp_async_wait<kStages - 2>();   // slab i has landed (this thread's copies)
        __syncthreads();                // ... everyone's; and slot (i-1) is free
        {
            const int nxt = i + kStages - 1;
            if (nxt < nloc) {
                const int kt = kt_begin + nxt;
                if (kt < interior_end) loader.load_interior(kt, nxt % kStages);
                else loader.load(kt, nxt % kStages, K, kt >= full_slabs);
            }
            cp_async_commit();
        }
        const float* a_s = sA + (i % kStages) * kAStage;
        const float* b_s = sB + (i % kStages) * kBStage;
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(a_s + k * kLdA + am);
            const float4 a1 = *reinterpret_cast<const float4*>(a_s + k * kLdA + am + kWM / 2);
            const float4 b0 = *reinterpret_cast<const float4*>(b_s + k * kLdB + bn);
            const float4 b1 = *reinterpret_cast<const float4*>(b_s + k * kLdB + bn + kWN / 2);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[ii][j] = fmaf(a[ii], b[j], acc[ii][j]);
        }
    }
    cp_async_wait<0>();

    if ((int)blockIdx.x >= dp_tiles) {
        // Split tile: publish this K range's partial, then let the last CTA
        // of the tile combine all of them.
        const int st = tile - dp_tiles;
        float* mine = partial + ((int64_t)st * splits + part) * (kBM * kBN);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = am + (i < 4 ? i : kWM / 2 + (i - 4));
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *reinterpret_cast<float4*>(mine + r * kBN + bn + h * (kWN / 2)) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(counters + st, 1u) == (unsigned)(splits - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const float* base = partial + (int64_t)st * splits * (kBM * kBN);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = am + (i < 4 ? i : kWM / 2 + (i - 4));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = r * kBN + bn + h * (kWN / 2);
                float4 sum = __ldcg(reinterpret_cast<const float4*>(base + c));
                for (int p = 1; p < splits; ++p) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(base + (int64_t)p * (kBM * kBN) + c));
                    sum.x += v.x, sum.y += v.y, sum.z += v.z, sum.w += v.w;
                }
                acc[i][4 * h] = sum.x, acc[i][4 * h + 1] = sum.y;
                acc[i][4 * h + 2] = sum.z, acc[i][4 * h + 3] = sum.w;
            }
        }
    }

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

int g_ctas_per_sm = kMinBlocks;

}  // namespace

cudaError_t ffma_setup() {
    cudaError_t e;
    if ((e = set_smem_attr<false, false>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<true, false>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<true, true>()) != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ffma_sgemm_kernel<true, true>, kThreads,
                                                      kSmemBytes);
    if (e != cudaSuccess) return e;
    g_ctas_per_sm = n > 0 ? n : 1;
    return cudaSuccess;
}

FfmaPlan ffma_plan(int M, int N, int K, int num_sms) {
    FfmaPlan p{};
    const int64_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = tiles_m * tiles_n;
    const int64_t slots = (int64_t)num_sms * g_ctas_per_sm;
    const int64_t nkt = (K + kBK - 1) / kBK;
    p.tiles = tiles;
    p.dp_tiles = tiles;
    p.splits = 1;
    const int64_t rem = slots > 0 ? tiles % slots : 0;
    // Split the tiles of a partial last wave along K, as many ways as still
    // fit in one wave, keeping at least kMinSlabs slabs per piece.
    constexpr int64_t kMinSlabs = 8;
    if (rem > 0) {
        int64_t s = slots / rem;
        if (s > nkt / kMinSlabs) s = nkt / kMinSlabs;
        if (s > 16) s = 16;
        if (s >= 2) {
            p.splits = (int)s;
            p.dp_tiles = tiles - rem;
            p.split_tiles = rem;
            p.partial_bytes = rem * s * kBM * kBN * (int64_t)sizeof(float);
            p.counter_bytes = rem * (int64_t)sizeof(unsigned);
        }
    }
    return p;
}

cudaError_t launch_ffma_sgemm(const float* A, const float* B, float* C, int M, int N, int K,
                              bool b_vec, bool c_vec, const FfmaPlan& plan, float* partial,
                              unsigned* counters, cudaStream_t stream) {
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    if (plan.tiles <= 0) return cudaSuccess;
    const int64_t ctas = plan.dp_tiles + plan.split_tiles * plan.splits;
    if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dim3 grid((unsigned)ctas), block(kThreads);
    const int dp = (int)plan.dp_tiles, sp = plan.splits;
#define LIBGEMM_FFMA_LAUNCH(BV, CV)                                                               \
    ffma_sgemm_kernel<BV, CV><<<grid, block, kSmemBytes, stream>>>(A, B, C, M, N, K, tiles_m,     \
                                                                    tiles_n, dp, sp, partial,     \
                                                                    counters)
    if (b_vec && c_vec) LIBGEMM_FFMA_LAUNCH(true, true);
    else if (b_vec) LIBGEMM_FFMA_LAUNCH(true, false);
    else if (c_vec) LIBGEMM_FFMA_LAUNCH(false, true);
    else LIBGEMM_FFMA_LAUNCH(false, false);
#undef LIBGEMM_FFMA_LAUNCH
    return cudaGetLastError();
}

}  // namespace libgemm
