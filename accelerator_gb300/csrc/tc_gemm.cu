// tc_gemm.cu -- tensor-core GEMM on sm_103a (modes GEMM_TF32, GEMM_BF16, GEMM_FP16).
//
// C_ij = sum_k A_ik B_kj ("Shared Memory Tiling for Matrix Multiplication",
// opening formula), A M x K row-major (K-major), B K x N row-major (N-major),
// C M x N row-major fp32.  The pages stop at naming tensor cores as the next
// step ("Matrix Multiplication -- Naive to Tiled", section 07, "Tensor Cores");
// this is that step written for the 5th-generation tensor cores.
//
// One persistent CTA per SM walks output tiles of 128 x 256.  Its six warps
// have fixed roles:
//   warp 0  TMA producer: one thread streams 128-byte-wide K slabs of A
//           (128 rows) and B (256 columns) into a 4-stage shared-memory ring
//           with cp.async.bulk.tensor; each slot has a "full" mbarrier that
//           the copy completes and an "empty" one the MMA frees.
//   warp 1  owns tensor memory (512 columns = two 128 x 256 fp32
//           accumulators) and one thread issues tcgen05.mma (M=128, N=256,
//           K=8 for TF32 / 16 for BF16), then tcgen05.commit to free the slot.
//   warps 2-5  epilogue: tcgen05.ld the finished accumulator (each warp its
//           32-lane quarter of TMEM), store fp32 rows of C guarded against M
//           and N, and hand the accumulator back.  With two accumulators the
//           epilogue of tile t overlaps the MMAs of tile t+1.
// The ring replaces the pages' two __syncthreads per tile (first page,
// section 05; second page's barrier discussion) by full/empty phases, and
// the TMA's zero fill of out-of-range boxes replaces their guarded loads.
//
// Shared-memory operand layouts (128-byte swizzle, each tile 1024-aligned):
//   A slab: 128 rows x 128 bytes of K, row r at r*128: the canonical K-major
//     layout, 8-row groups 1024 bytes apart (stride byte offset 1024).  The
//     k-th MMA of a slab starts 32*k bytes into the rows.
//   B slab: 128/es columns of N per 128-byte row, one row per k, boxes of
//     128/es columns side by side every (K rows * 128) bytes: the canonical
//     MN-major layout with leading byte offset = box size.  16-bit elements:
//     16-byte swizzle chunks, stride byte offset 1024 (8 k-rows); 32-bit
//     (TF32) elements: 32-byte swizzle chunks, stride byte offset 512 (4
//     k-rows).  The k-th MMA starts k*UMMA_K rows down.  B is read as the
//     caller stores it (K x N rows) in every mode.
//
// Every wait is bounded (see mbar_wait): if one expires the CTA records a
// timeout in the device error word, the roles stop, in-flight copies and
// MMAs are drained with bounded waits, TMEM is freed and the CTA returns.
#include <cstdlib>
#include <cstring>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace libgemm {
namespace {

constexpr int kBM = 128, kBN = 256;
constexpr int kStages = 4;
constexpr int kSlabBytes = 128;                      // K bytes per stage (one swizzle row)
constexpr int kABytes = kBM * kSlabBytes;            // 16 KB
constexpr int kBBytes = kBN * kSlabBytes;            // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = kBN;                        // fp32 accumulator columns per tile
constexpr int kTmemCols = 2 * kAccCols;              // 512
constexpr int kThreads = 192;
constexpr int kGroupM = 8;
constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

template <TcMode MODE>
struct Traits;
template <>
struct Traits<TcMode::kBF16> {
    static constexpr int kEs = 2;
    static constexpr uint32_t kFormat = 1;       // BF16
    static constexpr TcKind kKind = TcKind::kF16;
    // MN-major B: 128-byte swizzle of 16-byte chunks, repeating every 8
    // k-rows (1024 bytes), the stride byte offset between 8-row groups.
    static constexpr uint32_t kBMnLayout = kLayoutSw128, kBMnSbo = 1024;
    static constexpr int kAtomRows = 8;   // k-rows per swizzle atom (8 x 128 bytes)
};
template <>
struct Traits<TcMode::kF16> {
    static constexpr int kEs = 2;
    static constexpr uint32_t kFormat = 0;       // F16
    static constexpr TcKind kKind = TcKind::kF16;
    static constexpr uint32_t kBMnLayout = kLayoutSw128, kBMnSbo = 1024;
    static constexpr int kAtomRows = 8;
};
template <>
struct Traits<TcMode::kTF32> {
    static constexpr int kEs = 4;
    static constexpr uint32_t kFormat = 2;       // TF32
    static constexpr TcKind kKind = TcKind::kTF32;
    // An MN-major operand of 32-bit elements is read in the 128-byte swizzle
    // of 32-byte chunks (what the TMA writes with
    // CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B), whose pattern repeats every 4
    // k-rows: 512 bytes between 4-row groups.  (With the 16-byte-chunk
    // swizzle an MN-major kind::tf32 operand reads as zeros.)
    static constexpr uint32_t kBMnLayout = kLayoutSw128Atom32, kBMnSbo = 512;
    static constexpr int kAtomRows = 4;   // k-rows per swizzle atom (4 x 128 bytes)
};

struct Sched {
    int tiles_m, tiles_n;
    __device__ __forceinline__ void coords(int tile, int& m0, int& n0) const {
        const int per_group = kGroupM * tiles_n;
        const int group = tile / per_group;
        const int first_m = group * kGroupM;
        const int gsize = min(tiles_m - first_m, kGroupM);
        m0 = (first_m + (tile % per_group) % gsize) * kBM;
        n0 = ((tile % per_group) / gsize) * kBN;
    }
};

// Drain wait: bounded by time only (ignores the abort flag).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// Applies the epilogue in place to one thread's 32 accumulator values: row
// `row` of C, columns col0 .. col0 + 31.  Only kind 2 reads C, and only inside
// M x N (16 bytes at a time when vec: C rows 16-byte aligned); values outside
// are never stored.
__device__ __forceinline__ void epilogue_row32(const Epilogue& e, uint32_t (&v)[32],
                                               const float* crow, const float* C, int row,
                                               int col0, int M, int N, bool vec) {
    if (e.kind == 0) return;
    if (e.kind == 2 && row < M) {
        if (vec && col0 + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                if (!GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 16)) continue;
                const float4 r = epilogue_apply4(
                    e,
                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])),
                    crow + col0 + j);
                v[j] = __float_as_uint(r.x), v[j + 1] = __float_as_uint(r.y);
                v[j + 2] = __float_as_uint(r.z), v[j + 3] = __float_as_uint(r.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N && GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 4))
                    v[j] = __float_as_uint(epilogue_apply(e, __uint_as_float(v[j]), crow + col0 + j));
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__fmul_rn(e.alpha, __uint_as_float(v[j])));
}

template <TcMode MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b, float* __restrict__ C, int M, int N,
                   int K, int tiles_m, int tiles_n, int c_vec, const Epilogue epi, unsigned* err,
                   uint64_t limit_ns) {
    using T = Traits<MODE>;
    constexpr int kKElems = kSlabBytes / T::kEs;          // K per stage: 64 bf16 / 32 tf32
    constexpr int kUmmaK = 32 / T::kEs;                   // K per MMA: 16 / 8
    constexpr int kMmaPerStage = kKElems / kUmmaK;        // 4
    constexpr int kBoxN = kSlabBytes / T::kEs;            // N per B box: 64 / 32
    constexpr int kBoxes = kBN / kBoxN;                   // 4 / 8
    constexpr uint32_t kBoxBytes = kKElems * kSlabBytes;  // 8 KB / 4 KB
    constexpr uint32_t kIdesc = make_idesc(T::kFormat, kBM, kBN, false, true);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sA = base;                                   // kStages x kABytes
    const uint32_t sB = base + kStages * kABytes;               // kStages x kBBytes
    uint8_t* ctrl = gbase + kStages * kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
    // bars: full[0..S), empty[S..2S), acc_full[2S..2S+2), acc_empty[2S+2..2S+4), drain[2S+4]
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kStages;
    const uint32_t accf0 = full0 + 16 * kStages, acce0 = accf0 + 16, drain_bar = acce0 + 16;
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ctrl + 8 * (2 * kStages + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (2 * kStages + 5) + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4 * 32);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_holder)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const Sched sched{tiles_m, tiles_n};
    const int ntiles = tiles_m * tiles_n;
    const int nk = (K + kKElems - 1) / kKElems;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t last_phase[kStages];
            bool used[kStages];
            for (int s = 0; s < kStages; ++s) used[s] = false, last_phase[s] = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                int m0, n0;
                sched.coords(tile, m0, n0);
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, err, limit_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    tma_load_2d(sA + stage * kABytes, &map_a, fb, kb * kKElems, m0);
#pragma unroll
                    for (int j = 0; j < kBoxes; ++j)
                        tma_load_2d(sB + stage * kBBytes + j * kBoxBytes, &map_b, fb,
                                    n0 + j * kBoxN, kb * kKElems);
                    used[stage] = true;
                    last_phase[stage] = phase;
                    if (++stage == kStages) stage = 0, phase ^= 1u;
                }
                if (!ok) break;
            }
            // Every copy this thread issued must have landed before the CTA exits.
            for (int s = 0; s < kStages; ++s)
                if (used[s] && !drain_wait(full0 + 8 * s, last_phase[s], limit_ns))
                    atomicOr(err, kErrTimeout);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
                const int buf = lt & 1;
                const uint32_t use_parity = (uint32_t)(lt >> 1) & 1u;
                if (!mbar_wait(acce0 + 8 * buf, use_parity ^ 1u, abort_flag, err, limit_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kAccCols);
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, err, limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tile = sA + stage * kABytes;
                    const uint32_t b_tile = sB + stage * kBBytes;
#pragma unroll
                    for (int kk = 0; kk < kMmaPerStage; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(a_tile + kk * 32, 16, 1024);
                        const uint64_t bdesc = smem_desc(b_tile + kk * kUmmaK * kSlabBytes,
                                                         kBoxBytes, T::kBMnSbo, T::kBMnLayout);
                        tc_mma<T::kKind>(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty0 + 8 * stage);   // slot is free once these MMAs are done
                    if (++stage == kStages) stage = 0, phase ^= 1u;
                }
                if (!ok) break;
                tc_commit(accf0 + 8 * buf);          // accumulator ready for the epilogue
            }
            // All MMAs this thread issued must be complete before TMEM is freed.
            tc_commit(drain_bar);
            if (!drain_wait(drain_bar, 0, limit_ns)) atomicOr(err, kErrTimeout);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
        const int row_in_tile = quarter * 32 + lane;
        int lt = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++lt) {
            int m0, n0;
            sched.coords(tile, m0, n0);
            const int buf = lt & 1;
            const uint32_t use_parity = (uint32_t)(lt >> 1) & 1u;
            int ok = 0;
            if (lane == 0) ok = mbar_wait(accf0 + 8 * buf, use_parity, abort_flag, err, limit_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = m0 + row_in_tile;
            float* crow = C + (int64_t)row * N;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kAccCols);
#pragma unroll 1
            for (int c = 0; c < kAccCols / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), v);
                tmem_ld_wait();
                const int col0 = n0 + c * 32;
                epilogue_row32(epi, v, crow, C, row, col0, M, N, c_vec != 0);
                if (row < M) {
                    if (c_vec && col0 + 32 <= N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            if (GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 16))
                                *reinterpret_cast<float4*>(crow + col0 + j) =
                                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < N && GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 4))
                                crow[col0 + j] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acce0 + 8 * buf);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// 2-SM version: a cluster of two CTAs (a "pair") computes a 256 x 256 tile
// with tcgen05.mma.cta_group::2 (M = 256, N = 256).  Each CTA holds its own
// 128 rows of A and its own 128 columns of B in shared memory, so per MMA an
// SM reads 4 KB of A and 4 KB of B instead of 4 + 8, and its TMA writes half
// the B bytes: the shared-memory traffic per MMA cycle that limits the 1-SM
// kernel is cut by a third.  The accumulator is split by rows: each CTA's
// TMEM holds its 128 rows x 256 fp32 columns, and each CTA's epilogue stores
// its own rows.
//
// Roles (both CTAs run the same code):
//   warp 0  producer: loads this CTA's A rows and B columns of each K slab;
//           the copies of BOTH CTAs complete on the leader's "full" barrier,
//           which the leader's producer arms with the bytes of the pair.
//   warp 1  allocates TMEM for the pair (collectively with the peer's warp 1);
//           in the leader (cluster rank 0) one thread issues the MMAs and
//           commits them to the "empty" barriers of both CTAs (multicast),
//           and to both CTAs' accumulator-full barriers after a tile.
//   warps 2-5  epilogue of this CTA's rows; each warp then arrives on the
//           leader's accumulator-empty barrier (count 8: 4 warps x 2 CTAs).
// Work units: pair tiles, or (tile, K range) pieces of the tiles a K split
// cuts up, whose raw partial sums go to a workspace for tile_reduce_kernel.
// Launched with programmatic stream serialisation: the set-up above the
// grid dependency wait overlaps the previous kernel; no global memory is
// touched before it.
constexpr int kPStages = 6;

// Pair tile p of the pair kernel's grouped raster: rows m0 .. m0 + 255,
// columns n0 .. n0 + 255 (consecutive tiles walk down kGroupM tile rows).
__device__ __forceinline__ void pair_coords(int p, int pairs_m, int tiles_n, int& m0, int& n0) {
    const int per_group = kGroupM * tiles_n;
    const int group = p / per_group;
    const int first_m = group * kGroupM;
    const int gsize = min(pairs_m - first_m, kGroupM);
    m0 = (first_m + (p % per_group) % gsize) * (2 * kBM);
    n0 = ((p % per_group) / gsize) * kBN;
}
// How the pair kernel writes C: TMA stores from swizzled staging (16-byte
// aligned C rows), 16-byte vector stores, or 4-byte stores.
enum : int { kStoreScalar = 0, kStoreVec = 1, kStoreTma = 2 };
constexpr int kPHalfN = kBN / 2;                     // B columns held per CTA
constexpr int kPABytes = kBM * kSlabBytes;           // 16 KB
constexpr int kPBBytes = kPHalfN * kSlabBytes;       // 16 KB
constexpr int kPStageBytes = kPABytes + kPBBytes;    // 32 KB
// Epilogue staging: per epilogue warp two 32 x 32 fp32 blocks (4 KB each),
// laid out with the 128-byte swizzle the TMA store expects.
constexpr int kPStageCBytes = 4 * 2 * 32 * 32 * 4;   // 32 KB
constexpr size_t kPSmemBytes =
    size_t(kPStages) * kPStageBytes + kPStageCBytes + 1024 + 256;

template <TcMode MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_c,
                        const __grid_constant__ CUtensorMap map_w, float* __restrict__ C, int M,
                        int N, int K, int pairs_m, int tiles_n, int c_mode, const Epilogue epi,
                        int splits, int k_per_split, int whole_tiles, int b_4d, unsigned* err,
                        uint64_t limit_ns) {
    using T = Traits<MODE>;
    constexpr int kKElems = kSlabBytes / T::kEs;          // K per stage: 64 bf16 / 32 tf32
    constexpr int kUmmaK = 32 / T::kEs;                   // K per MMA: 16 / 8
    constexpr int kMmaPerStage = kKElems / kUmmaK;        // 4
    constexpr int kBoxN = kSlabBytes / T::kEs;            // N per MN-major B box: 64 (bf16)
    constexpr int kBoxes = kPHalfN / kBoxN;               // 2 (bf16)
    constexpr uint32_t kBoxBytes = kKElems * kSlabBytes;  // 8 KB (bf16)
    // The other B layout (b_4d): swizzle atoms of kAtomRows k-rows x 128
    // bytes ordered [k group][column block], so that the B operand of one
    // MMA (kUmmaK rows of all kBoxes column blocks) is 4 KB in one piece;
    // one 4-D TMA box per stage writes it.  Leading byte offset = one atom
    // (the next column block), stride byte offset = kBoxes atoms (the next
    // k group).
    constexpr uint32_t kAtomBytes = T::kAtomRows * kSlabBytes;            // 512 / 1024
    constexpr uint32_t kKGroupBytes = kBoxes * kAtomBytes;                // 2 KB
    constexpr uint32_t kMmaBBytes = (kUmmaK / T::kAtomRows) * kKGroupBytes;   // 4 KB
    constexpr uint32_t kIdesc = make_idesc(T::kFormat, 2 * kBM, kBN, false, true);
    constexpr uint32_t kPairTx = 2u * kPStageBytes;       // bytes the leader's full barrier awaits

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sA = base;                                   // kPStages x kPABytes
    const uint32_t sB = base + kPStages * kPABytes;             // kPStages x kPBBytes
    const uint32_t sC = base + kPStages * kPStageBytes;         // epilogue staging
    uint8_t* ctrl = gbase + kPStages * kPStageBytes + kPStageCBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
    // full[0..S), empty[S..2S), acc_full[2S..2S+2), acc_empty[2S+2..2S+4), drain[2S+4]
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kPStages;
    const uint32_t accf0 = full0 + 16 * kPStages, acce0 = accf0 + 16, drain_bar = acce0 + 16;
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ctrl + 8 * (2 * kPStages + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (2 * kPStages + 5) + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();            // 0: leader, 1: peer
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 2 * 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_holder)), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers and TMEM exist before anyone signals the other
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above touched only this cluster's shared memory and TMEM, so
    // it may overlap the end of the previous kernel on the stream; from here
    // on global memory (A, B, C, the workspace) is read and written.
    grid_dependency_wait();

    const int npairs = pairs_m * tiles_n;
    const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int nk = (K + kKElems - 1) / kKElems;
    // Work units: the first whole_tiles pair tiles whole (unit u is tile u,
    // all K), then each remaining tile as `splits` units over K slabs
    // [kb0, kb1).  A split unit stores its raw partial sum as one 256 x 256
    // block of the workspace map_w describes: block (tile - whole_tiles) *
    // splits + split, rows block * 256 .. +255.
    const int kps = splits > 1 ? k_per_split : nk;
    const int nunits = whole_tiles + (npairs - whole_tiles) * splits;
    // the pair tile p covers rows pm*256 .. +255 and columns pn*256 .. +255
    auto coords = [&](int p, int& m0, int& n0) { pair_coords(p, pairs_m, tiles_n, m0, n0); };
    // split = -1: a whole tile (stored to C); otherwise the workspace block
    auto unit = [&](int u, int& m0, int& n0, int& kb0, int& kb1, int& split) {
        if (u < whole_tiles) {
            coords(u, m0, n0);
            kb0 = 0, kb1 = nk, split = -1;
            return;
        }
        const int v = u - whole_tiles, t = v / splits;
        coords(whole_tiles + t, m0, n0);
        kb0 = (v - t * splits) * kps;
        kb1 = min(nk, kb0 + kps);
        split = v;   // workspace block index
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            const uint32_t full_leader0 = mapa_shared(full0, 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t last_phase[kPStages];
            bool used[kPStages];
            for (int s = 0; s < kPStages; ++s) used[s] = false, last_phase[s] = 0;
            for (int u = cluster_id; u < nunits; u += nclusters) {
                int m0, n0, kb0, kb1, split;
                unit(u, m0, n0, kb0, kb1, split);
                const int my_m0 = m0 + (int)rank * kBM, my_n0 = n0 + (int)rank * kPHalfN;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, err, limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, kPairTx);
                    const uint32_t fb = full_leader0 + 8 * stage;
                    tma_load_2d_pair(sA + stage * kPABytes, &map_a, fb, kb * kKElems, my_m0);
                    if (b_4d) {
                        tma_load_4d_pair(sB + stage * kPBBytes, &map_b, fb, 0, 0, my_n0 / kBoxN,
                                         kb * (kKElems / T::kAtomRows));
                    } else {
#pragma unroll
                        for (int j = 0; j < kBoxes; ++j)
                            tma_load_2d_pair(sB + stage * kPBBytes + j * kBoxBytes, &map_b, fb,
                                             my_n0 + j * kBoxN, kb * kKElems);
                    }
                    used[stage] = true;
                    last_phase[stage] = phase;
                    if (++stage == kPStages) stage = 0, phase ^= 1u;
                }
                if (!ok) break;
            }
            // every load of this CTA is issued: the next kernel (the split
            // fix-up) may be scheduled now; it waits for this grid to finish
            grid_launch_dependents();
            // Each copy issued here must have landed before the CTA exits: a
            // slot's copy has been consumed once the MMAs that read it freed it.
            for (int s = 0; s < kPStages; ++s)
                if (used[s] && !drain_wait(empty0 + 8 * s, last_phase[s], limit_ns))
                    atomicOr(err, kErrTimeout);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader CTA only) ----------------
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            for (int u = cluster_id; u < nunits; u += nclusters, ++lt) {
                int m0, n0, kb0, kb1, split;
                unit(u, m0, n0, kb0, kb1, split);
                const int buf = lt & 1;
                const uint32_t use_parity = (uint32_t)(lt >> 1) & 1u;
                if (!mbar_wait(acce0 + 8 * buf, use_parity ^ 1u, abort_flag, err, limit_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kAccCols);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, err, limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tile = sA + stage * kPABytes;
                    const uint32_t b_tile = sB + stage * kPBBytes;
#pragma unroll
                    for (int kk = 0; kk < kMmaPerStage; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(a_tile + kk * 32, 16, 1024);
                        const uint64_t bdesc =
                            b_4d ? smem_desc(b_tile + kk * kMmaBBytes, kAtomBytes, kKGroupBytes,
                                             T::kBMnLayout)
                                 : smem_desc(b_tile + kk * kUmmaK * kSlabBytes, kBoxBytes,
                                             T::kBMnSbo, T::kBMnLayout);
                        tc_mma_pair<T::kKind>(d_tmem, adesc, bdesc, kIdesc,
                                              (kb != kb0 || kk != 0) ? 1u : 0u);
                    }
                    tc_commit_pair_multicast(empty0 + 8 * stage, 0x3);   // frees the slot in both CTAs
                    if (++stage == kPStages) stage = 0, phase ^= 1u;
                }
                if (!ok) break;
                tc_commit_pair_multicast(accf0 + 8 * buf, 0x3);          // both epilogues may read
            }
            tc_commit_pair(drain_bar);
            if (!drain_wait(drain_bar, 0, limit_ns)) atomicOr(err, kErrTimeout);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t acce_leader0 = mapa_shared(acce0, 0);
        int stored = 0;   // TMA stores issued by this warp (lane 0's count, shared)
        int lt = 0;
        for (int u = cluster_id; u < nunits; u += nclusters, ++lt) {
            int m0, n0, kb0, kb1, split;
            unit(u, m0, n0, kb0, kb1, split);
            const int buf = lt & 1;
            const uint32_t use_parity = (uint32_t)(lt >> 1) & 1u;
            int ok = 0;
            if (lane == 0) ok = mbar_wait(accf0 + 8 * buf, use_parity, abort_flag, err, limit_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row0 = m0 + (int)rank * kBM + quarter * 32;   // this warp's 32 rows
            const int row = row0 + lane;
            float* crow = C + (int64_t)row * N;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kAccCols);
            // a split unit stores raw partials, always through TMA, into its block
            const bool to_ws = split >= 0;
            const int mode_u = to_ws ? kStoreTma : c_mode;
            const int ws_row0 = split * (2 * kBM) + (int)rank * kBM + quarter * 32;
#pragma unroll 1
            for (int c = 0; c < kAccCols / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), v);
                tmem_ld_wait();
                const int col0 = n0 + c * 32;
                if (!to_ws && mode_u != kStoreScalar)
                    epilogue_row32(epi, v, crow, C, row, col0, M, N, true);
                if (mode_u == kStoreTma) {
                    // Stage the warp's 32 x 32 block (row = lane) with the 128-byte
                    // swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)), then
                    // one lane writes it with a TMA store that clips at M and N.
                    const uint32_t stg = sC + (uint32_t)((quarter * 2 + (stored & 1)) * 4096);
                    if (stored >= 2) {
                        if (lane == 0) bulk_wait_group_read<1>();   // this buffer's last store has read it
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), v[4 * j],
                                     v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0 && row0 < M && col0 < N) {
                        if (to_ws)
                            tma_store_2d(&map_w, stg, c * 32, ws_row0);
                        else
                            tma_store_2d(&map_c, stg, col0, row0);
                        bulk_commit_group();
                        ++stored;
                    }
                    stored = __shfl_sync(0xffffffffu, stored, 0);
                } else if (mode_u == kStoreScalar) {
                    // C rows not 16-byte aligned: stage the block (row = lane) as
                    // above, then write it a row at a time, lane j to column
                    // col0 + j, so that each store (and the epilogue's read of C)
                    // covers 128 contiguous bytes instead of 32 rows.
                    const uint32_t stg = sC + (uint32_t)(quarter * 2 * 4096);
                    if (lane == 0) bulk_wait_group_read<0>();   // no TMA store still reads it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), v[4 * j],
                                     v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    __syncwarp();
                    const int col = col0 + lane;
#pragma unroll 4
                    for (int i = 0; i < 32; ++i) {
                        const int r = row0 + i;
                        if (r >= M) break;   // the same for the whole warp
                        const float x = ld_shared_f32(
                            stg + (uint32_t)(i * 128 + ((((lane >> 2) ^ (i & 7))) << 4) + (lane & 3) * 4));
                        float* dst = C + (int64_t)r * N + col;
                        if (col < N && GEMM_DBG_OK(dst, C, (int64_t)M * N * 4, 4))
                            *dst = epilogue_apply(epi, x, dst);
                    }
                    __syncwarp();   // the block is read before the next chunk overwrites it
                } else if (row < M) {
                    if (mode_u == kStoreVec && col0 + 32 <= N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            if (GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 16))
                                *reinterpret_cast<float4*>(crow + col0 + j) =
                                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < N && GEMM_DBG_OK(crow + col0 + j, C, (int64_t)M * N * 4, 4))
                                crow[col0 + j] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader0 + 8 * buf);
        }
        if (lane == 0) bulk_wait_group<0>();   // every store of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no more signals or MMAs between the two CTAs after this
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// K-split fix-up of the pair kernel: for each split tile t (pair tiles
// whole_tiles + t), C := epilogue(sum of workspace blocks t * splits + s,
// s = 0 .. splits - 1, added in that order: the same sum on every run).  A
// thread handles four columns of one row; four blocks' loads are issued
// before they are added.
__global__ void __launch_bounds__(256)
    tile_reduce_kernel(const float* __restrict__ ws, int splits, int whole_tiles, int split_tiles,
                       int pairs_m, int tiles_n, float* __restrict__ C, int M, int N, int c_vec,
                       const Epilogue epi) {
    constexpr int kTile = 2 * kBM;                        // 256 x 256 blocks
    constexpr int64_t kPerTile = (int64_t)kTile * (kTile / 4);
    constexpr int64_t kBlock = (int64_t)kTile * kTile;
    const int64_t units = (int64_t)split_tiles * kPerTile;
    grid_dependency_wait();   // the MMA kernel's partials are complete and visible
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(u / kPerTile);
        const int r = (int)((u % kPerTile) / (kTile / 4)), c4 = (int)(u % (kTile / 4));
        int m0, n0;
        pair_coords(whole_tiles + t, pairs_m, tiles_n, m0, n0);
        const int i = m0 + r, j = n0 + 4 * c4;
        if (i >= M || j >= N) continue;
        const float* p = ws + ((int64_t)t * splits * kTile + r) * kTile + 4 * c4;
        const int64_t ws_bytes = (int64_t)split_tiles * splits * kBlock * 4;
        if (!GEMM_DBG_OK(p, ws, ws_bytes, 16) || !GEMM_DBG_OK(p + (splits - 1) * kBlock, ws, ws_bytes, 16))
            continue;
        float4 acc = __ldcg(reinterpret_cast<const float4*>(p));
        int sp = 1;
        for (; sp + 4 <= splits; sp += 4) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[q] = __ldcg(reinterpret_cast<const float4*>(p + (sp + q) * kBlock));
#pragma unroll
            for (int q = 0; q < 4; ++q)
                acc.x += v[q].x, acc.y += v[q].y, acc.z += v[q].z, acc.w += v[q].w;
        }
        for (; sp < splits; ++sp) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p + sp * kBlock));
            acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
        }
        float* c = C + (int64_t)i * N + j;
        if (!GEMM_DBG_OK(c, C, (int64_t)M * N * 4, c_vec ? 16 : 4)) continue;
        if (c_vec) {   // N % 4 == 0: the four columns are inside C
            *reinterpret_cast<float4*>(c) = epilogue_apply4(epi, acc, c);
        } else {
            const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j + q < N) c[q] = epilogue_apply(epi, a[q], c + q);
        }
    }
}

}  // namespace

TcShape tc_shape(TcMode mode) {
    const int es = mode == TcMode::kTF32 ? 4 : 2;
    return TcShape{kBM, kBN, kSlabBytes / es, kSlabBytes / es, mode == TcMode::kTF32 ? 4 : 8,
                   kPHalfN / (kSlabBytes / es)};
}


template <TcMode MODE>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes);
}

template <TcMode MODE>
static cudaError_t set_pair_attr() {
    return cudaFuncSetAttribute(tc_gemm_pair_kernel<MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmemBytes);
}

// Clusters of two that can be resident at once (0: pairs unavailable).
static int g_max_pairs = 0;
// GEMM_FORCE_CONFIG=b_boxes_2d: B always in the per-column-block layout.
static bool g_force_b2d = false;

bool tc_b_atoms(TcMode mode, int64_t K, int64_t N, int64_t ldb) {
    const TcShape s = tc_shape(mode);
    return g_max_pairs > 0 && !g_force_b2d && ldb == N && N % s.b_box_n == 0 &&
           K % s.b_atom_rows == 0;
}

template <TcMode MODE>
static int query_max_pairs(int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t tc_setup() {
    cudaError_t e;
    if ((e = set_attr<TcMode::kBF16>()) != cudaSuccess) return e;
    if ((e = set_attr<TcMode::kTF32>()) != cudaSuccess) return e;
    if ((e = set_attr<TcMode::kF16>()) != cudaSuccess) return e;
    if ((e = set_pair_attr<TcMode::kBF16>()) != cudaSuccess) return e;
    if ((e = set_pair_attr<TcMode::kF16>()) != cudaSuccess) return e;
    if ((e = set_pair_attr<TcMode::kTF32>()) != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int a = query_max_pairs<TcMode::kBF16>(sms);
    const int b = query_max_pairs<TcMode::kTF32>(sms);
    g_max_pairs = a < b ? a : b;
    // GEMM_FORCE_CONFIG=single_cta: use the 1-SM kernel even where pairs fit
    // (it is otherwise only taken on devices that cannot hold pair clusters).
    const char* force = std::getenv("GEMM_FORCE_CONFIG");
    if (force && std::strcmp(force, "single_cta") == 0) g_max_pairs = 0;
    g_force_b2d = force && std::strcmp(force, "b_boxes_2d") == 0;
    return cudaSuccess;
}

int tc_max_pairs() { return g_max_pairs; }

// K split of the pair kernel, from a cost model in units of one K slab of one
// pair tile (about 0.33 us in either mode: 2*256*256*64 BF16 or 2*256*256*32
// TF32 FLOP at 1/76 of the tensor rate), with R = rounds of clusters:
//   unsplit     R(pairs) * (nk + overhead)
//   all split   R(pairs * S) * (ceil(nk / S) + overhead) + reduce
//   tail split  the tiles of a partial last round cut S ways so that they
//               fill one round: R(whole) * (nk + overhead) + ceil(nk / S) +
//               overhead + reduce
// where reduce = a launch plus the workspace blocks (256 KB per tile and
// split) written and read and C written, at about 2 MB per slab time
// (~6 TB/s), or 4 MB when the workspace is small enough to stay in L2.
// A split must save 1 - kMinGain and keep >= kMinSplitSlabs slabs a unit.
// (Measured at 4096^3 and 8192^3, the tail split gains 1-2 %: less than the
// model says, since a partly filled last round runs faster per cluster.)
TcSplit tc_plan_split(TcMode mode, int64_t M, int64_t N, int64_t K) {
    constexpr double kUnitOverhead = 4.0, kReduceFixed = 6.0, kL2Bytes = 96.0e6;
    constexpr double kMinGain = 0.98, kBlockBytes = 256.0 * 256.0 * 4.0;
    constexpr int kMinSplitSlabs = 4, kMaxSplits = 128;
    constexpr double kMaxWorkspace = 512.0 * 1024 * 1024;
    const int es = mode == TcMode::kTF32 ? 4 : 2;
    const int64_t kel = kSlabBytes / es;
    const int64_t nk = (K + kel - 1) / kel;
    const int64_t pairs = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + kBN - 1) / kBN);
    const int64_t clusters = g_max_pairs;
    if (clusters <= 0 || pairs <= 0 || nk < 2 * kMinSplitSlabs) return kNoSplit;
    auto rounds = [&](int64_t units) { return (double)((units + clusters - 1) / clusters); };
    auto reduce = [&](int64_t tiles, int64_t S) {
        const double ws = (double)tiles * S * kBlockBytes;
        const double per_slab = ws <= kL2Bytes ? 4.0e6 : 2.0e6;
        return kReduceFixed + (double)tiles * (2.0 * S + 1.0) * kBlockBytes / per_slab;
    };
    const double unsplit = rounds(pairs) * ((double)nk + kUnitOverhead);
    double best = kMinGain * unsplit;
    TcSplit plan = kNoSplit;
    const int64_t rem = pairs % clusters, whole = pairs - rem;
    for (int64_t S = 2; S <= kMaxSplits && S * kMinSplitSlabs <= nk; ++S) {
        const int64_t kps = (nk + S - 1) / S;
        if ((nk + kps - 1) / kps != S) continue;   // every unit must have a slab
        if (pairs < clusters) {                     // all tiles split
            if ((double)pairs * S * kBlockBytes > kMaxWorkspace) break;
            const double cost = rounds(pairs * S) * ((double)kps + kUnitOverhead) + reduce(pairs, S);
            if (cost < best) best = cost, plan = TcSplit{(int)S, (int)kps, 0};
        } else if (rem > 0 && rem * S <= clusters) {   // the last round's tiles split
            if ((double)rem * S * kBlockBytes > kMaxWorkspace) break;
            const double cost = rounds(whole) * ((double)nk + kUnitOverhead) +
                                ((double)kps + kUnitOverhead) + reduce(rem, S);
            if (cost < best) best = cost, plan = TcSplit{(int)S, (int)kps, (int)whole};
        }
    }
    return plan;
}

cudaError_t launch_tc_gemm_pair(TcMode mode, const CUtensorMap& map_a,
                                const CUtensorMap& map_b, const CUtensorMap* map_c,
                                const CUtensorMap* map_w, float* C, int M, int N, int K, bool c_vec,
                                const Epilogue& epi, const TcSplit& split, bool b_atoms,
                                unsigned* err, uint64_t limit_ns, cudaStream_t stream) {
    const int pairs_m = (M + 2 * kBM - 1) / (2 * kBM), tiles_n = (N + kBN - 1) / kBN;
    const int64_t pairs = (int64_t)pairs_m * tiles_n;
    if (pairs <= 0) return cudaSuccess;
    if (pairs > 0x3FFFFFFF || g_max_pairs <= 0) return cudaErrorInvalidValue;
    const bool splitting = split.splits > 1;
    const int sp = splitting ? split.splits : 1;
    const int64_t whole = splitting ? split.whole_tiles : pairs;
    // split units store raw partials through TMA into the workspace map_w
    if (splitting && (!map_w || whole < 0 || whole >= pairs || split.k_per_split < 1))
        return cudaErrorInvalidValue;
    const int64_t units = whole + (pairs - whole) * sp;
    if (units > 0x3FFFFFFF) return cudaErrorInvalidValue;
    const int clusters = (int)(units < g_max_pairs ? units : g_max_pairs);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kUsePdl ? 2 : 1;
    const int cm = map_c ? kStoreTma : (c_vec ? kStoreVec : kStoreScalar);
    const CUtensorMap& mc = map_c ? *map_c : map_a;   // unused unless cm == kStoreTma
    const CUtensorMap& mw = map_w ? *map_w : map_a;   // unused without split units
    const int kps = splitting ? split.k_per_split : 0, wt = (int)whole;
    const int b4 = b_atoms ? 1 : 0;
    cudaError_t e;
    if (mode == TcMode::kBF16)
        e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<TcMode::kBF16>, map_a, map_b, mc, mw, C, M,
                               N, K, pairs_m, tiles_n, cm, epi, sp, kps, wt, b4, err, limit_ns);
    else if (mode == TcMode::kTF32)
        e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<TcMode::kTF32>, map_a, map_b, mc, mw, C, M,
                               N, K, pairs_m, tiles_n, cm, epi, sp, kps, wt, b4, err, limit_ns);
    else
        e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<TcMode::kF16>, map_a, map_b, mc, mw, C, M,
                               N, K, pairs_m, tiles_n, cm, epi, sp, kps, wt, b4, err, limit_ns);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int64_t tc_split_workspace_bytes(const TcSplit& split, int64_t M, int64_t N) {
    if (split.splits < 2) return 0;
    const int64_t pairs = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + kBN - 1) / kBN);
    return (pairs - split.whole_tiles) * split.splits * (int64_t)(2 * kBM) * (2 * kBM) * 4;
}

cudaError_t launch_tc_tile_reduce(const float* ws, const TcSplit& split, float* C, int M, int N,
                                  bool c_vec, const Epilogue& epi, int num_sms,
                                  cudaStream_t stream) {
    const int pairs_m = (M + 2 * kBM - 1) / (2 * kBM), tiles_n = (N + kBN - 1) / kBN;
    const int64_t pairs = (int64_t)pairs_m * tiles_n;
    const int64_t split_tiles = pairs - split.whole_tiles;
    if (split.splits < 2 || split_tiles <= 0 || split.whole_tiles < 0) return cudaErrorInvalidValue;
    const int64_t units = split_tiles * (2 * kBM) * (2 * kBM / 4);
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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, tile_reduce_kernel, ws, split.splits,
                                             split.whole_tiles, (int)split_tiles, pairs_m, tiles_n,
                                             C, M, N, c_vec ? 1 : 0, epi);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_tc_gemm(TcMode mode, const CUtensorMap& map_a,
                           const CUtensorMap& map_b, float* C, int M, int N, int K, bool c_vec,
                           const Epilogue& epi, int num_sms, unsigned* err, uint64_t limit_ns,
                           cudaStream_t stream) {
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = (int64_t)tiles_m * tiles_n;
    if (tiles <= 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    const int cv = c_vec ? 1 : 0;
#define LIBGEMM_TC_LAUNCH(MODE_)                                                              \
    tc_gemm_kernel<MODE_><<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, C, M, N, K, tiles_m, \
                                                                  tiles_n, cv, epi, err, limit_ns)
    if (mode == TcMode::kBF16)
        LIBGEMM_TC_LAUNCH(TcMode::kBF16);
    else if (mode == TcMode::kF16)
        LIBGEMM_TC_LAUNCH(TcMode::kF16);
    else
        LIBGEMM_TC_LAUNCH(TcMode::kTF32);
#undef LIBGEMM_TC_LAUNCH
    return cudaGetLastError();
}

LIBGEMM_DEBUG_READER(tc_debug_flags)

}  // namespace libgemm
