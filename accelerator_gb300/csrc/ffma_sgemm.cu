// ffma_sgemm.cu -- exact binary32 GEMM on the CUDA cores (mode GEMM_FP32).
//
// C_ij = sum_k A_ik B_kj ("Shared Memory Tiling for Matrix Multiplication",
// opening formula), row-major as in "Matrix Multiplication -- Naive to
// Tiled", section 02.  Every C_ij is one chain of fused multiply-adds with k
// ascending, so the result is the sequential binary32 sum of exact products
// (when the tiles do not fill the GPU -- fewer than one wave, or a partial
// last wave -- the sum, in order, of such chains over consecutive K ranges:
// added in the kernel by the last CTA of a split tile after a full wave, or
// by splitk_reduce_kernel from whole M x N partial blocks otherwise).
//
// Design (GB300 rather than the pages' 16x16/32x32 tiles):
//   * A CTA owns a 128 x 128 tile of C and each thread a TM x TN register
//     block, made of 4 x 4 sub-blocks so that every fragment is one 128-bit
//     shared-memory load -- the register blocking of "From 306 ms to 86 ms"
//     (4 x 4 there) and of "Further Optimisation Ideas" on the first page,
//     taken further.  The lanes of a warp are laid out so that each
//     quarter-warp reads at most two distinct 16-byte chunks of one operand:
//     such a 128-bit load costs two shared-memory wavefronts instead of four.
//   * K is walked in slabs of 16 through a multi-stage ring of shared-memory
//     buffers filled by cp.async, so global loads of later slabs overlap the
//     arithmetic on the current one (the page's "double buffering", deeper).
//   * The A slab is stored transposed (k-major, [k][m], padded by 4 floats) so
//     that 4 consecutive rows of A at one k are one 128-bit load; the
//     element-wise copies that do the transposition are arranged so a warp's
//     32 stores hit 32 different banks.  B slabs are copied 16 bytes at a time
//     when rows are 16-byte aligned, else 4 bytes at a time.
//   * Tiles wholly inside M and N copy their slabs without any check; edge
//     tiles and the last, partial slab zero-fill out-of-range elements
//     (source size 0) and store only in-range C elements -- the boundary
//     handling of the first page's section 05, for any M, K, N.
//   * Tiles are visited in groups of 16 tile-rows so CTAs running together
//     share A and B slabs in L2 (at 4096^3 a wave of 456 tiles then spans
//     16 rows and ~29 columns of tiles, ~90 MB of operands: DRAM reads per
//     launch 271 MB, against 325 MB with groups of 8 and 472 MB with 32;
//     the time is the same, the kernel being bound by its FMA pipe).
#include <cstdlib>
#include <cstring>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace libgemm {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16;
constexpr int kPadA = 4;
constexpr int kLdA = kBM + kPadA;               // floats per k-row of the A slab
constexpr int kLdB = kBN;
constexpr int kAStage = kBK * kLdA;             // floats
constexpr int kBStage = kBK * kLdB;
constexpr int kGroupM = 16;

// A thread-tile layout.  LM x LN lanes per warp, each lane TM x TN outputs
// (TM/4 row chunks LM*4 apart, TN/4 column chunks LN*4 apart); kNMajor puts
// consecutive lanes along N (ln = lane % LN) instead of along M.
template <int TM_, int TN_, int LM_, int LN_, bool kNMajor_, int THREADS_, int STAGES_, int MINB_>
struct Cfg {
    static constexpr int TM = TM_, TN = TN_, LM = LM_, LN = LN_;
    static constexpr bool kNMajor = kNMajor_;
    static constexpr int kThreads = THREADS_, kStages = STAGES_, kMinBlocks = MINB_;
    static constexpr int WM = LM * TM, WN = LN * TN;             // warp tile
    static constexpr int kWarpsM = kBM / WM, kWarpsN = kBN / WN;
    static constexpr size_t kSmemBytes = size_t(kStages) * (kAStage + kBStage) * sizeof(float);
    static_assert(LM * LN == 32, "a warp is 32 lanes");
    static_assert(kWarpsM * kWarpsN * 32 == kThreads, "warps cover the tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "4 x 4 sub-blocks");
};
// 16 x 8 per thread, 128 threads, lanes 4 (M) x 8 (N) with N fastest: a
// quarter-warp shares one A chunk, so 6 fragment loads per k cost 16
// wavefronts for 128 FMAs (an 8 x 8 layout with lanes 8 (M) x 4 (N): 12 for
// 64; measured 19 % slower at 4096^3).
using Cfg16x8 = Cfg<16, 8, 4, 8, true, 128, 3, 3>;
using FfmaCfg = Cfg16x8;

// The copies of one thread, planned once per tile so that issuing the copies
// of a K slab is a few pointer and address additions.
//
// A: kBM x kBK elements, kAPer per thread.  A pass covers 8 consecutive k of
// THREADS/8 rows; lanes 0-7 take one row, so a warp reads 4 x 32 contiguous
// bytes and its transposed stores land in banks (4*k + row) mod 32, all
// distinct.  B: rows of kBN columns copied 16 bytes (kBVec) or 4 bytes per
// copy, a warp covering one contiguous 512- or 128-byte row piece.
template <bool kBVec, int THREADS>
struct SlabLoader {
    static constexpr int kRowsPerPass = THREADS / 8;               // rows of A per pass
    static constexpr int kARowGroups = kBM / kRowsPerPass;
    static constexpr int kAPer = (kBM * kBK) / THREADS;            // copies of A per thread
    static constexpr int kBElems = kBVec ? 4 : 1;                  // floats per B copy
    static constexpr int kBPerRow = kBN / kBElems;                 // copies per B row
    static constexpr int kBRowsPerPass = THREADS / kBPerRow;
    static constexpr int kBPer = kBK / kBRowsPerPass;              // copies of B per thread
    static_assert(kAPer == kARowGroups * (kBK / 8), "A split");
    static_assert(THREADS % kBPerRow == 0 && kBK % kBRowsPerPass == 0, "B split");

    const float* a_base;               // A itself: source of zero-size copies
    const float* a_ptr;                // &A[m0 + tid/8][tid % 8]
    const float* b_ptr;                // &B[tid / kBPerRow][n0 + column of this thread]
    int64_t a_group_step;              // kRowsPerPass * K: to the next row group of A
    int64_t n;                         // the row stride of B (ldb >= N; with the
                                       // vector copies, a chunk that crosses N reads
                                       // the row's padding up to ldb)
    uint32_t a_row_ok;                 // bit j: row group j of this thread is < M
    bool b_col_ok;
    int a_k, b_k;                      // this thread's k offset within a slab (A, B)
    uint32_t a_dst, b_dst;             // shared addresses in ring slot 0
#ifdef GEMM_DEBUG
    const float *dbg_a, *dbg_b;        // the operands and their sizes in bytes
    int64_t dbg_a_bytes, dbg_b_bytes;
#endif

    __device__ __forceinline__ SlabLoader(const float* A, const float* B, float* sA, float* sB,
                                          int M, int N, int K, int ldb, int m0, int n0, int tid) {
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
        b_ptr = b_col_ok ? B + (int64_t)b_k * ldb + n0 + bc : B;
        n = ldb;
        b_dst = smem_u32(sB + b_k * kLdB + bc);
#ifdef GEMM_DEBUG
        dbg_a = A, dbg_b = B;
        dbg_a_bytes = (int64_t)M * K * 4, dbg_b_bytes = (int64_t)K * ldb * 4;
#endif
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
            for (int g = 0; g < kBK / 8; ++g)
                if (GEMM_DBG_OK(row + 8 * g, dbg_a, dbg_a_bytes, 4))
                    cp_async_4(adst + (uint32_t)((8 * g * kLdA + kRowsPerPass * j) * 4), row + 8 * g);
        }
        const uint32_t bdst = b_dst + (uint32_t)(slot * kBStage * 4);
        const float* bsrc = b_ptr + (int64_t)k0 * n;
#pragma unroll
        for (int r = 0; r < kBPer; ++r) {
            const float* src = bsrc + (int64_t)(kBRowsPerPass * r) * n;
            const uint32_t dst = bdst + (uint32_t)(kBRowsPerPass * r * kLdB * 4);
            if (!GEMM_DBG_OK(src, dbg_b, dbg_b_bytes, 4 * kBElems)) continue;
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
            if (ok) ok = GEMM_DBG_OK(src, dbg_a, dbg_a_bytes, 4);
            cp_async_4(adst + (uint32_t)((8 * g * kLdA + kRowsPerPass * j) * 4), src, ok);
        }
        const uint32_t bdst = b_dst + (uint32_t)(slot * kBStage * 4);
        const float* bsrc = b_ptr + (int64_t)k0 * n;
#pragma unroll
        for (int r = 0; r < kBPer; ++r) {
            bool ok = b_col_ok;
            if (check_k) ok = ok && (k0 + kBRowsPerPass * r + b_k < K);
            const float* src = ok ? bsrc + (int64_t)(kBRowsPerPass * r) * n : b_ptr;
            if (ok) ok = GEMM_DBG_OK(src, dbg_b, dbg_b_bytes, 4 * kBElems);
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
template <class CF, bool kBVec, bool kCVec, bool kWide>
__global__ void __launch_bounds__(CF::kThreads, CF::kMinBlocks)
    ffma_sgemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K, int ldb, int tiles_m, int tiles_n,
                      int dp_tiles, int splits, float* __restrict__ partial,
                      unsigned* __restrict__ counters, const Epilogue epi) {
    constexpr int TM = CF::TM, TN = CF::TN, kStages = CF::kStages;
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
    const int wm0 = (warp / CF::kWarpsN) * CF::WM;
    const int wn0 = (warp % CF::kWarpsN) * CF::WN;
    const int lm = CF::kNMajor ? lane / CF::LN : lane % CF::LM;
    const int ln = CF::kNMajor ? lane % CF::LN : lane / CF::LM;
    const int am = wm0 + lm * 4;               // row chunks am + c*LM*4, c < TM/4
    const int bn = wn0 + ln * 4;               // column chunks bn + c*LN*4, c < TN/4
    // row / column (in the tile) of the i-th / j-th element of this thread's block
    auto row_of = [&](int i) { return am + (i / 4) * (CF::LM * 4) + (i % 4); };
    auto col_of = [&](int j) { return bn + (j / 4) * (CF::LN * 4) + (j % 4); };

    // Accumulators in pairs of rows: acc2[p][j] = (C[2p][j], C[2p+1][j]) of this
    // thread's block, updated with packed two-lane FMAs (each lane one
    // round-to-nearest FMA, exactly as the scalar instruction).
    float2 acc2[TM / 2][TN];
#pragma unroll
    for (int p = 0; p < TM / 2; ++p)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc2[p][j] = make_float2(0.0f, 0.0f);
    auto acc = [&](int i, int j) -> float& { return (i & 1) ? acc2[i >> 1][j].y : acc2[i >> 1][j].x; };

    const SlabLoader<kBVec, CF::kThreads> loader(A, B, sA, sB, M, N, K, kBVec ? ldb : N, m0, n0, tid);
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
            float2 a2[TM / 2];
            float b[TN];
#pragma unroll
            for (int c = 0; c < TM / 4; ++c) {
                const float4 t = *reinterpret_cast<const float4*>(a_s + k * kLdA + am + c * CF::LM * 4);
                a2[2 * c] = make_float2(t.x, t.y), a2[2 * c + 1] = make_float2(t.z, t.w);
            }
#pragma unroll
            for (int c = 0; c < TN / 4; ++c) {
                const float4 t = *reinterpret_cast<const float4*>(b_s + k * kLdB + bn + c * CF::LN * 4);
                b[4 * c] = t.x, b[4 * c + 1] = t.y, b[4 * c + 2] = t.z, b[4 * c + 3] = t.w;
            }
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float2 bj = make_float2(b[j], b[j]);
#pragma unroll
                for (int pp = 0; pp < TM / 2; ++pp) acc2[pp][j] = __ffma2_rn(a2[pp], bj, acc2[pp][j]);
            }
        }
    }
    cp_async_wait<0>();

    if constexpr (kWide) {
        // Wide split (every CTA a piece): `partial` is a workspace of
        // `splits` M x N blocks; store this K range's raw partial into block
        // `part` as if it were C (a separate kernel adds the blocks in order).
        C = partial + (int64_t)part * M * N;
    } else if ((int)blockIdx.x >= dp_tiles) {
        // Split tile: publish this K range's partial, then let the last CTA
        // of the tile combine all of them.
        const int st = tile - dp_tiles;
        float* mine = partial + ((int64_t)st * splits + part) * (kBM * kBN);
#ifdef GEMM_DEBUG
        const int64_t part_bytes = (int64_t)(tiles_m * tiles_n - dp_tiles) * splits * (kBM * kBN) * 4;
#endif
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int h = 0; h < TN / 4; ++h)
                if (GEMM_DBG_OK(mine + row_of(i) * kBN + col_of(4 * h), partial, part_bytes, 16))
                    *reinterpret_cast<float4*>(mine + row_of(i) * kBN + col_of(4 * h)) =
                        make_float4(acc(i, 4 * h), acc(i, 4 * h + 1), acc(i, 4 * h + 2), acc(i, 4 * h + 3));
        __threadfence();
        __syncthreads();
        if (tid == 0)
            s_last = GEMM_DBG_OK(counters + st, counters, (int64_t)(tiles_m * tiles_n - dp_tiles) * 4, 4) &&
                     atomicAdd(counters + st, 1u) == (unsigned)(splits - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const float* base = partial + (int64_t)st * splits * (kBM * kBN);
#pragma unroll
        for (int i = 0; i < TM; ++i) {
#pragma unroll
            for (int h = 0; h < TN / 4; ++h) {
                const int c = row_of(i) * kBN + col_of(4 * h);
                if (!GEMM_DBG_OK(base + (int64_t)(splits - 1) * (kBM * kBN) + c, partial, part_bytes, 16) ||
                    !GEMM_DBG_OK(base + c, partial, part_bytes, 16))
                    continue;
                float4 sum = __ldcg(reinterpret_cast<const float4*>(base + c));
                for (int p = 1; p < splits; ++p) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(base + (int64_t)p * (kBM * kBN) + c));
                    sum.x += v.x, sum.y += v.y, sum.z += v.z, sum.w += v.w;
                }
                acc(i, 4 * h) = sum.x, acc(i, 4 * h + 1) = sum.y;
                acc(i, 4 * h + 2) = sum.z, acc(i, 4 * h + 3) = sum.w;
            }
        }
    }

    // Store the block: guarded against M and N.
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + row_of(i);
        if (row >= M) continue;
        float* crow = C + (int64_t)row * N;
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
            const int col = n0 + col_of(4 * h);
            if (kCVec && col < N) {   // N % 4 == 0: all four columns are in range
                if (!GEMM_DBG_OK(crow + col, C, (int64_t)M * N * 4, 16)) continue;
                *reinterpret_cast<float4*>(crow + col) = epilogue_apply4(
                    epi,
                    make_float4(acc(i, 4 * h), acc(i, 4 * h + 1), acc(i, 4 * h + 2),
                                acc(i, 4 * h + 3)),
                    crow + col);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < N && GEMM_DBG_OK(crow + col + j, C, (int64_t)M * N * 4, 4))
                        crow[col + j] = epilogue_apply(epi, acc(i, 4 * h + j), crow + col + j);
            }
        }
    }
}

// ---- stream-K form: one persistent CTA per resident slot ----
// For shapes whose tiles fill between half a wave and two waves of CTA
// slots, whole tiles leave slots idle (2048^3: 256 tiles on 456 slots run as
// 104 SMs with two CTAs and 48 with one) or a last wave partly empty.  Here
// the space of tile x K-slab units (tiles in raster order, slabs ascending
// within a tile) is cut into gridDim.x equal contiguous ranges, one per CTA,
// [total * b / G, total * (b + 1) / G).  A CTA walks its range tile by tile,
// each tile as the FFMA chain over its slabs of the range (the loop of
// ffma_sgemm_kernel); a tile it covers wholly is stored to C with the
// epilogue; the first and the last tile of its range, when it covers only
// part of them, store their raw partial sums to workspace blocks 2b and
// 2b + 1 (kBM x kBN floats each) and count the piece on the tile's counter;
// the CTA that stores a tile's last piece (in time) adds all of its pieces
// in K order and stores C: C_ij is then ((p0 + p1) + p2), the same on every
// run.  With at least half a wave of tiles a CTA's range is longer than
// half a tile, so a tile has at most three pieces (kMaxPieces); with a
// quarter to half a wave it can have up to five, and the pieces past the
// third are added one by one after them, still in K order.

// Tile coordinates in the grouped raster (kGroupM tile-rows per group).
__device__ __forceinline__ void ffma_tile_coords(int tile, int tiles_m, int tiles_n, int& m0,
                                                 int& n0) {
    const int per_group = kGroupM * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * kGroupM;
    const int gsize = min(tiles_m - first_m, kGroupM);
    m0 = (first_m + (tile % per_group) % gsize) * kBM;
    n0 = ((tile % per_group) / gsize) * kBN;
}

// First unit of CTA b's range, and the CTA whose range holds unit x.
__device__ __forceinline__ int64_t stream_lo(int64_t total, int64_t b, int64_t G) {
    return total * b / G;
}
__device__ __forceinline__ int64_t stream_owner(int64_t total, int64_t x, int64_t G) {
    return ((x + 1) * G - 1) / total;
}

constexpr int kMaxPieces = 3;

template <class CF, bool kBVec, bool kCVec>
__global__ void __launch_bounds__(CF::kThreads, CF::kMinBlocks)
    ffma_stream_kernel(const float* __restrict__ A, const float* __restrict__ B,
                       float* __restrict__ C, int M, int N, int K, int ldb, int tiles_m, int tiles_n,
                       float* __restrict__ ws, unsigned* __restrict__ counters,
                       const Epilogue epi) {
    constexpr int TM = CF::TM, TN = CF::TN, kStages = CF::kStages;
    extern __shared__ __align__(16) float smem[];
    float* sA = smem;
    float* sB = smem + kStages * kAStage;
    __shared__ unsigned s_last;

    const int nkt = (K + kBK - 1) / kBK;
    const int64_t G = gridDim.x;
    const int64_t total = (int64_t)tiles_m * tiles_n * nkt;
    const int64_t lo = stream_lo(total, blockIdx.x, G), hi = stream_lo(total, blockIdx.x + 1, G);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm0 = (warp / CF::kWarpsN) * CF::WM;
    const int wn0 = (warp % CF::kWarpsN) * CF::WN;
    const int lm = CF::kNMajor ? lane / CF::LN : lane % CF::LM;
    const int ln = CF::kNMajor ? lane % CF::LN : lane / CF::LM;
    const int am = wm0 + lm * 4;
    const int bn = wn0 + ln * 4;
    auto row_of = [&](int i) { return am + (i / 4) * (CF::LM * 4) + (i % 4); };
    auto col_of = [&](int j) { return bn + (j / 4) * (CF::LN * 4) + (j % 4); };
    const int full_slabs = K / kBK;
#ifdef GEMM_DEBUG
    const int64_t ws_bytes = G * 2 * (kBM * kBN) * 4;
#endif

    for (int64_t u = lo; u < hi;) {
        const int tile = (int)(u / nkt);
        const int kt_begin = (int)(u - (int64_t)tile * nkt);
        const int kt_end = (int)(hi - u < (int64_t)(nkt - kt_begin) ? kt_begin + (hi - u) : nkt);
        int m0, n0;
        ffma_tile_coords(tile, tiles_m, tiles_n, m0, n0);

        float2 acc2[TM / 2][TN];
#pragma unroll
        for (int p = 0; p < TM / 2; ++p)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc2[p][j] = make_float2(0.0f, 0.0f);
        auto acc = [&](int i, int j) -> float& {
            return (i & 1) ? acc2[i >> 1][j].y : acc2[i >> 1][j].x;
        };

        const SlabLoader<kBVec, CF::kThreads> loader(A, B, sA, sB, M, N, K, kBVec ? ldb : N, m0, n0, tid);
        const int nloc = kt_end - kt_begin;
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
            cp_async_wait<kStages - 2>();
            __syncthreads();
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
                float2 a2[TM / 2];
                float b[TN];
#pragma unroll
                for (int c = 0; c < TM / 4; ++c) {
                    const float4 t =
                        *reinterpret_cast<const float4*>(a_s + k * kLdA + am + c * CF::LM * 4);
                    a2[2 * c] = make_float2(t.x, t.y), a2[2 * c + 1] = make_float2(t.z, t.w);
                }
#pragma unroll
                for (int c = 0; c < TN / 4; ++c) {
                    const float4 t =
                        *reinterpret_cast<const float4*>(b_s + k * kLdB + bn + c * CF::LN * 4);
                    b[4 * c] = t.x, b[4 * c + 1] = t.y, b[4 * c + 2] = t.z, b[4 * c + 3] = t.w;
                }
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const float2 bj = make_float2(b[j], b[j]);
#pragma unroll
                    for (int pp = 0; pp < TM / 2; ++pp)
                        acc2[pp][j] = __ffma2_rn(a2[pp], bj, acc2[pp][j]);
                }
            }
        }
        cp_async_wait<0>();

        if (kt_begin == 0 && kt_end == nkt) {
            // the whole tile in this range: C, with the epilogue, guarded
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int row = m0 + row_of(i);
                if (row >= M) continue;
                float* crow = C + (int64_t)row * N;
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    const int col = n0 + col_of(4 * h);
                    if (kCVec && col < N) {
                        if (!GEMM_DBG_OK(crow + col, C, (int64_t)M * N * 4, 16)) continue;
                        *reinterpret_cast<float4*>(crow + col) = epilogue_apply4(
                            epi,
                            make_float4(acc(i, 4 * h), acc(i, 4 * h + 1), acc(i, 4 * h + 2),
                                        acc(i, 4 * h + 3)),
                            crow + col);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (col + j < N && GEMM_DBG_OK(crow + col + j, C, (int64_t)M * N * 4, 4))
                                crow[col + j] = epilogue_apply(epi, acc(i, 4 * h + j), crow + col + j);
                    }
                }
            }
        } else {
            // a piece: the raw partial of the whole kBM x kBN block
            float* blk = ws + ((int64_t)blockIdx.x * 2 + (u == lo ? 0 : 1)) * (kBM * kBN);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    float* p = blk + row_of(i) * kBN + col_of(4 * h);
                    if (GEMM_DBG_OK(p, ws, ws_bytes, 16))
                        *reinterpret_cast<float4*>(p) =
                            make_float4(acc(i, 4 * h), acc(i, 4 * h + 1), acc(i, 4 * h + 2),
                                        acc(i, 4 * h + 3));
                }
            // count the piece; the last one to arrive adds the tile's pieces
            const int64_t x0 = (int64_t)tile * nkt;
            const int64_t b0 = stream_owner(total, x0, G), b1 = stream_owner(total, x0 + nkt - 1, G);
            const int npieces = (int)(b1 - b0 + 1);
            __threadfence();
            __syncthreads();
            // the counters' zero fill (the launch before this one, which may
            // still run: programmatic stream serialisation) is complete and visible
            grid_dependency_wait();
            if (tid == 0)
                s_last = GEMM_DBG_OK(counters + tile, counters, (int64_t)tiles_m * tiles_n * 4, 4) &&
                         atomicAdd(counters + tile, 1u) == (unsigned)(npieces - 1);
            __syncthreads();
            if (s_last) {
                __threadfence();
                // the pieces' blocks in K order: the tile is the first piece of
                // CTA b's range unless that range began before it
                const float* pb[kMaxPieces];
#pragma unroll
                for (int q = 0; q < kMaxPieces; ++q) {
                    const int64_t b = b0 + q < b1 ? b0 + q : b1;
                    pb[q] = ws + (2 * b + (b == b0 && stream_lo(total, b, G) < x0 ? 1 : 0)) *
                                     (int64_t)(kBM * kBN);
                }
                // eight fragments at a time, every piece's loads issued before the
                // adds (pieces beyond kMaxPieces, which only ranges shorter than
                // half a tile make, are added one by one after them, in K order)
#pragma unroll
                for (int f0 = 0; f0 < TM * (TN / 4); f0 += 8) {
                    float4 v[kMaxPieces][8];
#pragma unroll
                    for (int q = 0; q < kMaxPieces; ++q)
#pragma unroll
                        for (int f = 0; f < 8; ++f) {
                            const int i = (f0 + f) / (TN / 4), h = (f0 + f) % (TN / 4);
                            const float* p = pb[q] + row_of(i) * kBN + col_of(4 * h);
                            v[q][f] = q < npieces && GEMM_DBG_OK(p, ws, ws_bytes, 16)
                                          ? __ldcg(reinterpret_cast<const float4*>(p))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                    for (int f = 0; f < 8; ++f) {
                        const int i = (f0 + f) / (TN / 4), h = (f0 + f) % (TN / 4);
                        float4 sum = v[0][f];
#pragma unroll
                        for (int q = 1; q < kMaxPieces; ++q)
                            if (q < npieces)
                                sum.x += v[q][f].x, sum.y += v[q][f].y, sum.z += v[q][f].z,
                                    sum.w += v[q][f].w;
                        for (int64_t b = b0 + kMaxPieces; b <= b1; ++b) {
                            const float* p =
                                ws + 2 * b * (int64_t)(kBM * kBN) + row_of(i) * kBN + col_of(4 * h);
                            if (!GEMM_DBG_OK(p, ws, ws_bytes, 16)) continue;
                            const float4 w = __ldcg(reinterpret_cast<const float4*>(p));
                            sum.x += w.x, sum.y += w.y, sum.z += w.z, sum.w += w.w;
                        }
                        const int row = m0 + row_of(i), col = n0 + col_of(4 * h);
                        if (row >= M) continue;
                        float* crow = C + (int64_t)row * N;
                        if (kCVec && col < N) {
                            if (GEMM_DBG_OK(crow + col, C, (int64_t)M * N * 4, 16))
                                *reinterpret_cast<float4*>(crow + col) =
                                    epilogue_apply4(epi, sum, crow + col);
                        } else {
                            const float a[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (col + j < N &&
                                    GEMM_DBG_OK(crow + col + j, C, (int64_t)M * N * 4, 4))
                                    crow[col + j] = epilogue_apply(epi, a[j], crow + col + j);
                        }
                    }
                }
            }
        }
        u += nloc;
        __syncthreads();   // every warp is done with the ring before the next tile refills it
    }
}

template <bool BV, bool CV>
cudaError_t set_smem_attr() {
    cudaError_t e = cudaFuncSetAttribute(ffma_sgemm_kernel<FfmaCfg, BV, CV, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FfmaCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(ffma_sgemm_kernel<FfmaCfg, BV, CV, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FfmaCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(ffma_stream_kernel<FfmaCfg, BV, CV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)FfmaCfg::kSmemBytes);
}

int g_ctas_per_sm = FfmaCfg::kMinBlocks;

}  // namespace

cudaError_t ffma_setup() {
    cudaError_t e;
    if ((e = set_smem_attr<false, false>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<false, true>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<true, false>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<true, true>()) != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ffma_sgemm_kernel<FfmaCfg, true, true, false>,
                                                      FfmaCfg::kThreads, FfmaCfg::kSmemBytes);
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
    // Fewer tiles than one wave holds: every tile is split (at least
    // kMinSlabsWide slabs a piece, one wave, at most 256 pieces and
    // kMaxWorkspace bytes of partials), each piece stores its partial as a
    // whole M x N block, and a second kernel adds the blocks in piece order.
    // (Its loads are independent of one another; the in-kernel combination,
    // kept for the split tiles of a last wave, is latency-bound: 2 splits of
    // a 256^3 product took 53 us in the kernel against 24 us this way.)
    constexpr int64_t kMinSlabsWide = 4, kMaxWorkspace = 512ll << 20;
    // Stream-K (below): one persistent CTA per slot, between a quarter of a
    // wave and two waves of tiles, with K long enough that a CTA's range
    // holds at least kMinStreamSlabs slabs (GEMM_FORCE_CONFIG=ffma_no_stream
    // disables it).
    constexpr int64_t kMinStreamSlabs = 32, kStreamCost = 8, kSplitCost = 8, kMinSlabs = 8;
    static const bool no_stream = [] {
        const char* f = std::getenv("GEMM_FORCE_CONFIG");
        return f && std::strcmp(f, "ffma_no_stream") == 0;
    }();
    const int64_t total = tiles * nkt;
    bool stream_k = !no_stream && slots > 0 && 4 * tiles > slots && tiles < 2 * slots &&
                    tiles % slots != 0 && total >= kMinStreamSlabs * slots;
    if (slots > 0 && tiles < slots && slots / tiles >= 2 && nkt >= 2 * kMinSlabsWide) {
        int64_t s = slots / tiles;
        if (s > nkt / kMinSlabsWide) s = nkt / kMinSlabsWide;
        if (s > 256) s = 256;
        const int64_t block = (int64_t)M * N * (int64_t)sizeof(float);
        if (s * block > kMaxWorkspace) s = kMaxWorkspace / block;
        // Below half a wave stream-K is taken instead when the split's s x
        // tiles CTAs would leave more than 7 % of the slots idle (889 x
        // 4037 x 2830: 606 -> 454 us; 1500 x 3000 x 1800: 400 -> 348 us);
        // where they fill the slots the split stays (1536 x 2048 x 1536: 186
        // against 192 us).
        const bool sk_instead = stream_k && s * tiles * 100 < slots * 93;
        if (s >= 2 && !sk_instead) {
            p.splits = (int)s;
            p.dp_tiles = 0;
            p.split_tiles = tiles;
            p.wide = true;
            p.ws_bytes = s * block;
            return p;
        }
    }
    // Stream-K under one wave is always taken (whole tiles leave slots
    // idle: 2048^3 365 -> 309 us, 2432^3 603 -> 498 us).  From one to two
    // waves it is taken when its cost in slab times, an equal share plus
    // kStreamCost (restarts and the partial tiles), is under 97 % of a full
    // wave plus the last wave as split below (its pieces plus kSplitCost):
    // measured 3072^3 1069 -> 977 us and 3584^3 1694 -> 1528 us taken; 2944^3
    // (tail split 6 ways, 850 against 866 us) and 3840^3 (1.97 waves, 1815
    // against 1863 us) left as they were.
    if (stream_k && tiles > slots) {
        int64_t s = slots / (tiles - slots);
        if (s > nkt / kMinSlabs) s = nkt / kMinSlabs;
        if (s > 16) s = 16;
        const int64_t tail = s >= 2 ? (nkt + s - 1) / s + kSplitCost : nkt;
        const int64_t cost = (total + slots - 1) / slots + kStreamCost;
        stream_k = cost * 100 < (nkt + tail) * 97;
    }
    if (stream_k) {
        p.stream = true;
        p.stream_ctas = slots;
        p.dp_tiles = 0;
        p.ws_bytes = p.stream_ctas * 2 * kBM * kBN * (int64_t)sizeof(float);   // two blocks a CTA
        p.counter_bytes = tiles * (int64_t)sizeof(unsigned);                    // one a tile
        return p;
    }
    // Split the tiles of a partial last wave (after at least one full wave)
    // along K, as many ways as still fit in one wave, keeping at least
    // kMinSlabs slabs per piece; the last piece of a tile adds them up.
    if (rem > 0 && tiles > slots) {
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

// Launches the variant for the operands' vector widths; the wide split has
// its own instantiation so that the other kernels compile as they would
// without it.
template <bool BV, bool CV>
static void launch_variant(dim3 grid, size_t smem, cudaStream_t stream, const float* A,
                           const float* B, float* C, int M, int N, int K, int ldb, int tiles_m,
                           int tiles_n, int dp, int sp, const FfmaPlan& plan, float* partial,
                           unsigned* counters, float* ws, const Epilogue& epi) {
    if (plan.wide)
        ffma_sgemm_kernel<FfmaCfg, BV, CV, true><<<grid, FfmaCfg::kThreads, smem, stream>>>(
            A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp, sp, ws, nullptr, kPlainStore);
    else
        ffma_sgemm_kernel<FfmaCfg, BV, CV, false><<<grid, FfmaCfg::kThreads, smem, stream>>>(
            A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp, sp, partial, counters, epi);
}

cudaError_t launch_ffma_sgemm(const float* A, const float* B, float* C, int M, int N, int K,
                              int ldb, bool b_vec, bool c_vec, const FfmaPlan& plan,
                              float* partial, unsigned* counters, const Epilogue& epi, float* ws,
                              cudaStream_t stream) {
    if (ldb < N || (b_vec && ldb % 4 != 0)) return cudaErrorInvalidValue;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    if (plan.tiles <= 0) return cudaSuccess;
    if (plan.stream) {
        if (!ws || !counters || plan.stream_ctas <= 0 || plan.stream_ctas > 0x7FFFFFFF)
            return cudaErrorInvalidValue;
        // Programmatic stream serialisation: the CTAs start while the zero
        // fill of the counters before them finishes; everything they read
        // before their first counter update (A, B) was written before it.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.stream_ctas);
        cfg.blockDim = dim3(FfmaCfg::kThreads);
        cfg.dynamicSmemBytes = FfmaCfg::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = kUsePdl ? 1 : 0;
        cudaError_t e;
        if (b_vec && c_vec)
            e = cudaLaunchKernelEx(&cfg, ffma_stream_kernel<FfmaCfg, true, true>, A, B, C, M, N, K, ldb,
                                   tiles_m, tiles_n, ws, counters, epi);
        else if (b_vec)
            e = cudaLaunchKernelEx(&cfg, ffma_stream_kernel<FfmaCfg, true, false>, A, B, C, M, N, K, ldb,
                                   tiles_m, tiles_n, ws, counters, epi);
        else if (c_vec)
            e = cudaLaunchKernelEx(&cfg, ffma_stream_kernel<FfmaCfg, false, true>, A, B, C, M, N, K, ldb,
                                   tiles_m, tiles_n, ws, counters, epi);
        else
            e = cudaLaunchKernelEx(&cfg, ffma_stream_kernel<FfmaCfg, false, false>, A, B, C, M, N,
                                   K, ldb, tiles_m, tiles_n, ws, counters, epi);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t ctas = plan.dp_tiles + plan.split_tiles * plan.splits;
    if (ctas > 0x7FFFFFFF || (plan.wide && !ws)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)ctas);
    const int dp = (int)plan.dp_tiles, sp = plan.splits;
    const size_t smem = FfmaCfg::kSmemBytes;
    if (b_vec && c_vec)
        launch_variant<true, true>(grid, smem, stream, A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp, sp,
                                   plan, partial, counters, ws, epi);
    else if (b_vec)
        launch_variant<true, false>(grid, smem, stream, A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp, sp,
                                    plan, partial, counters, ws, epi);
    else if (c_vec)
        launch_variant<false, true>(grid, smem, stream, A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp, sp,
                                    plan, partial, counters, ws, epi);
    else
        launch_variant<false, false>(grid, smem, stream, A, B, C, M, N, K, ldb, tiles_m, tiles_n, dp,
                                     sp, plan, partial, counters, ws, epi);
    return cudaGetLastError();
}

LIBGEMM_DEBUG_READER(ffma_debug_flags)

}  // namespace libgemm
