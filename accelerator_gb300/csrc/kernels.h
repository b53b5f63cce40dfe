// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not installed; callers use include/gemm.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace libgemm {

// Launch the tensor-core kernel and the split fix-ups with programmatic
// stream serialization, so that their set-up overlaps the end of the kernel
// before them (each waits for that kernel before touching global memory).
constexpr bool kUsePdl = true;

// What every kernel does with a finished sum acc of C_ij:
//   kind 0  C_ij := acc                          (C is not read)
//   kind 1  C_ij := alpha * acc, rounded once    (C is not read)
//   kind 2  C_ij := fma(beta, C_ij, alpha * acc), alpha * acc rounded first
// -- the generalised product C = alpha*A*B + beta*C of the cuBLAS call in
// "Matrix Multiplication -- Naive to Tiled", section 07.
struct Epilogue {
    float alpha, beta;
    int kind;
};
constexpr Epilogue kPlainStore{1.0f, 0.0f, 0};

#ifdef __CUDACC__
__device__ __forceinline__ float epilogue_apply(const Epilogue& e, float acc, const float* c) {
    if (e.kind == 0) return acc;
    const float t = __fmul_rn(e.alpha, acc);
    return e.kind == 1 ? t : __fmaf_rn(e.beta, *c, t);
}
// Four consecutive elements; c must be 16-byte aligned when e.kind == 2.
__device__ __forceinline__ float4 epilogue_apply4(const Epilogue& e, float4 acc, const float* c) {
    if (e.kind == 0) return acc;
    float4 t = make_float4(__fmul_rn(e.alpha, acc.x), __fmul_rn(e.alpha, acc.y),
                           __fmul_rn(e.alpha, acc.z), __fmul_rn(e.alpha, acc.w));
    if (e.kind == 2) {
        const float4 o = *reinterpret_cast<const float4*>(c);
        t = make_float4(__fmaf_rn(e.beta, o.x, t.x), __fmaf_rn(e.beta, o.y, t.y),
                        __fmaf_rn(e.beta, o.z, t.z), __fmaf_rn(e.beta, o.w, t.w));
    }
    return t;
}
#endif

// ---- exact-FP32 CUDA-core GEMM (ffma_sgemm.cu) ----
// b_vec: B rows may be copied 16 bytes at a time (N % 4 == 0, B 16-byte aligned).
// c_vec: C rows may be stored 16 bytes at a time (N % 4 == 0, C 16-byte aligned).
// Work split: the first dp_tiles tiles whole, the last split_tiles tiles each
// in `splits` K ranges whose partials (partial_bytes of scratch) are summed by
// the last CTA of the tile (counter_bytes of zeroed counters).
// Wide plan (wide = true): every tile is split; the pieces store their raw
// partials into ws_bytes of workspace (splits blocks of M x N floats) and
// launch_splitk_reduce adds them and applies the epilogue.
// Stream-K plan (stream = true): stream_ctas persistent CTAs share the tile x
// K-slab units equally; ws_bytes of workspace hold two partial tiles per CTA,
// and counter_bytes of counters (one per tile, zeroed before the launch) let
// the last piece of a split tile add the pieces up (`counters` argument).
struct FfmaPlan {
    int64_t tiles, dp_tiles, split_tiles;
    int splits;
    int64_t partial_bytes, counter_bytes;
    bool wide;
    int64_t ws_bytes;
    bool stream;
    int64_t stream_ctas;
};
cudaError_t ffma_setup();
FfmaPlan ffma_plan(int M, int N, int K, int num_sms);
cudaError_t launch_ffma_sgemm(const float* A, const float* B, float* C, int M, int N, int K,
                              int ldb, bool b_vec, bool c_vec, const FfmaPlan& plan,
                              float* partial, unsigned* counters, const Epilogue& epi, float* ws,
                              cudaStream_t stream);


// ---- small-product FFMA GEMM (ffma_small.cu) ----
// Products with at most kSmallMaxMN outputs and K <= kSmallMaxK take the
// 32 x 32-tile kernel (one launch, no K split); GEMM_FORCE_CONFIG=ffma_small
// or =ffma_tiles128 makes every FP32 product take one of the two kernels
// (testing and tuning only).
constexpr int64_t kSmallMaxMN = 384 * 384, kSmallMaxK = 512;
bool ffma_small_fits(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_ffma_small(const float* A, const float* B, float* C, int M, int N, int K,
                              bool b_vec, bool c_vec, const Epilogue& epi, cudaStream_t stream);
unsigned ffma_small_debug_flags();

// ---- tcgen05 tensor-core GEMM (tc_gemm.cu) ----
enum class TcMode { kBF16, kTF32, kF16 };
struct TcShape {
    int block_m, block_n;   // output tile per CTA
    int k_elems;            // K elements per pipeline stage (128 bytes)
    int b_box_n;            // N extent of one TMA box of B (128 bytes)
    int b_atom_rows;        // k-rows per swizzle atom of B (4 TF32, 8 BF16/FP16)
    int b_blocks;           // B column blocks (of b_box_n) per CTA of a pair
};
TcShape tc_shape(TcMode mode);
cudaError_t tc_setup();
// Clusters of two CTAs of the 2-SM kernel that fit at once (0: unavailable).
int tc_max_pairs();
// 2-SM (CTA pair) kernel, B read MN-major in every mode.  Its TMA boxes: A
// as for the 1-SM kernel (block_m rows x 128 bytes); B, 128-byte swizzle of
// 16-byte chunks for 16-bit elements and of 32-byte chunks for TF32, either
// as 2-D boxes of k_elems rows x 128 bytes (b_box_n columns), or with
// b_atoms as one 4-D box per stage over the view (b_box_n columns, b_atom_rows
// k-rows, N / b_box_n column blocks, K / b_atom_rows k groups) of B, box
// (b_box_n, b_atom_rows, b_blocks, k_elems / b_atom_rows): each MMA's B
// operand then lies in one piece (tc_b_atoms says when that form applies).
// map_c (may be null): C as a 2-D fp32 tensor, box 32 x 32, 128-byte swizzle,
// for TMA stores of the epilogue; without it C is stored by the threads.
// K split of the pair kernel: the first whole_tiles pair tiles (in the
// kernel's raster order) are computed whole into C; every later tile as
// `splits` units of k_per_split K slabs (k_elems each; the last unit takes
// the rest, and every unit has at least one), each storing its raw partial
// as one 256 x 256 fp32 block of a workspace (block (tile - whole_tiles) *
// splits + split), which launch_tc_tile_reduce adds up into C.
// Bounds-check flags of each translation unit's kernels, read and cleared
// (debug build; always 0 in the release build).
unsigned ffma_debug_flags();
unsigned tc_debug_flags();
unsigned prep_debug_flags();

struct TcSplit {
    int splits, k_per_split, whole_tiles;
};
constexpr TcSplit kNoSplit{1, 0, 0};
// The split the pair kernel should use for an M x K x N product (kNoSplit
// when splitting would not pay).
TcSplit tc_plan_split(TcMode mode, int64_t M, int64_t N, int64_t K);
// Workspace bytes a split needs (0 for kNoSplit).
int64_t tc_split_workspace_bytes(const TcSplit& split, int64_t M, int64_t N);
// map_w (needed when split.splits > 1): the workspace as a 2-D fp32 tensor of
// 256 columns, row stride 256, box 32 x 32, 128-byte swizzle.
cudaError_t launch_tc_gemm_pair(TcMode mode, const CUtensorMap& map_a,
                                const CUtensorMap& map_b, const CUtensorMap* map_c,
                                const CUtensorMap* map_w, float* C, int M, int N, int K, bool c_vec,
                                const Epilogue& epi, const TcSplit& split, bool b_atoms,
                                unsigned* err, uint64_t limit_ns, cudaStream_t stream);
// Whether the pair kernel reads B (row stride ldb elements) in the
// atom-ordered 4-D form: pairs available, B read in place with N a multiple
// of b_box_n and K of b_atom_rows (so the 4-D view covers B exactly), and not
// disabled by GEMM_FORCE_CONFIG=b_boxes_2d.
bool tc_b_atoms(TcMode mode, int64_t K, int64_t N, int64_t ldb);
// C := the epilogue applied to the sum, in split order, of the workspace
// blocks of every split tile (the whole tiles are left as they are).
cudaError_t launch_tc_tile_reduce(const float* ws, const TcSplit& split, float* C, int M, int N,
                                  bool c_vec, const Epilogue& epi, int num_sms, cudaStream_t stream);
// C (M x N) := the epilogue applied to the sum, in split order, of the
// partials ws[s * ws_rows + i][j] (row stride ws_ld floats).
cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t ws_rows, int64_t ws_ld,
                                 float* C, int64_t M, int64_t N, bool c_vec, const Epilogue& epi,
                                 int num_sms, cudaStream_t stream);
// 1-SM kernel (128 x 256 tiles), the fallback where pair clusters do not fit.
cudaError_t launch_tc_gemm(TcMode mode, const CUtensorMap& map_a,
                           const CUtensorMap& map_b, float* C, int M, int N, int K, bool c_vec,
                           const Epilogue& epi, int num_sms, unsigned* err, uint64_t limit_ns,
                           cudaStream_t stream);

// ---- helpers (prep.cu) ----
// Copy a rows x cols matrix of es-byte elements from row stride src_ld to
// row stride dst_ld (both in elements).
cudaError_t launch_restride(const void* src, void* dst, int64_t rows, int64_t cols,
                            int64_t src_ld, int64_t dst_ld, int es, cudaStream_t stream);
// dst (rows x cols bfloat16, row stride dst_ld elements) = round-to-nearest-
// even of src (rows x cols float, dense).
cudaError_t launch_to_bf16(const float* src, void* dst, int64_t rows, int64_t cols,
                           int64_t dst_ld, cudaStream_t stream);
// Both operands of GEMM_FP32_VIA_BF16 in one launch when their rows allow
// 16-byte loads (cols % 4 == 0, 16-byte aligned src, ld % 4 == 0), else two
// launch_to_bf16 calls; *launches receives the number of kernels enqueued.
cudaError_t launch_to_bf16_pair(const float* a, void* a_dst, int64_t a_rows, int64_t a_cols,
                                int64_t a_ld, const float* b, void* b_dst, int64_t b_rows,
                                int64_t b_cols, int64_t b_ld, cudaStream_t stream, int* launches);
// GEMM_TF32_RN: both operands rounded to TF32 (to nearest, ties away from
// zero; binary32 with the 13 low fraction bits zero) into rows of stride
// a_ld / b_ld floats, one launch when both operands' rows allow 16-byte
// loads and stores, else one element-wise launch each.
cudaError_t launch_to_tf32_pair(const float* a, float* a_dst, int64_t a_rows, int64_t a_cols,
                                int64_t a_ld, const float* b, float* b_dst, int64_t b_rows,
                                int64_t b_cols, int64_t b_ld, cudaStream_t stream, int* launches);
cudaError_t launch_fill_zero(float* C, int64_t n, cudaStream_t stream);
// C := beta * C over n elements, each rounded once (beta != 0).
cudaError_t launch_scale(float* C, int64_t n, float beta, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream);

// ---- host-side hooks of the C ABI (api.cu) ----
// Per-device set-up of the library (device check, kernel attributes, error
// word); returns a gemm_status code.
int device_setup(int* num_sms, unsigned** err);
// How a tensor-core product (TF32, BF16, FP16 mode) runs: the row strides
// its kernels read A and B with, the K split, and the device scratch that
// takes, as one block [re-strided A | re-strided B | split workspace], each
// part a multiple of 256 bytes.  gemm() takes the block from its memory
// pool; gemm_tf32_noalloc() from its static buffer.
struct TcPlan {
    TcMode mode;
    bool pad_a, pad_b;            // operand copied into scratch with a 16-byte row stride
    int64_t lda, ldb;             // row strides (elements) the kernels read A and B with
    int64_t a_bytes, b_bytes;     // scratch for the copies (0: read in place)
    TcSplit split;
    int64_t ws_bytes;             // split workspace (0: the product is not split)
    int64_t scratch_bytes() const { return a_bytes + b_bytes + ws_bytes; }
};
TcPlan tc_plan(TcMode mode, const void* A, const void* B, int64_t M, int64_t K, int64_t N);
// Enqueues a planned product (K > 0) on `stream`; scratch: plan.scratch_bytes()
// bytes of device memory, 256-byte aligned (may be null when that is 0).
// Returns a gemm_status code.
int tc_product(const TcPlan& plan, const void* A, const void* B, float* C, int64_t M, int64_t K,
               int64_t N, const Epilogue& epi, void* scratch, cudaStream_t stream);
// Add one to the library's launch counter.
void count_launch();

}  // namespace libgemm
