// api.cu -- the C ABI of libgemm (include/gemm.h): argument checks, the
// per-device set-up, the choice of kernel and of a K split, TMA descriptors,
// stream-ordered scratch (re-strided or rounded operands, split workspaces),
// and the device error word.  Host code only, apart from the error word.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm.h"
#include "debug.cuh"
#include "kernels.h"

namespace {

using namespace libgemm;

// One per device (a __device__ variable exists once per device context).
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s for any single pipeline wait

struct DeviceState {
    std::atomic<bool> done{false};   // set-up finished (read without the lock)
    bool ready = false;
    int status = GEMM_OK;
    int num_sms = 0;
    unsigned* err = nullptr;
    // Scratch comes from this pool, stream-ordered.  It keeps what it has
    // reserved (release threshold: never), so repeated calls reuse memory
    // instead of mapping it afresh after every synchronisation.
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool make_pool(int dev, cudaMemPool_t* pool) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(pool, &props) != cudaSuccess) return false;
    uint64_t keep = UINT64_MAX;
    return cudaMemPoolSetAttribute(*pool, cudaMemPoolAttrReleaseThreshold, &keep) == cudaSuccess;
}

// Per-device set-up, once: device check, SM count, error word address,
// kernel attributes, and the driver's tensor-map encoder.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    DeviceState& st = g_dev[dev];
    if (st.done.load(std::memory_order_acquire)) {   // every later call: no lock
        *out = &st;
        return st.status;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st.ready) {
        st.ready = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            st.status = GEMM_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            st.status = GEMM_ERR_UNSUPPORTED_DEVICE;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), g_error_word) != cudaSuccess ||
                   ffma_setup() != cudaSuccess || tc_setup() != cudaSuccess) {
            st.status = GEMM_ERR_CUDA;
        } else if (!make_pool(dev, &st.pool)) {
            st.status = GEMM_ERR_CUDA;
        } else if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                st.status = GEMM_ERR_CUDA;
            else
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        if (st.status != GEMM_OK) cudaGetLastError();   // do not leave a stale error behind
        st.done.store(true, std::memory_order_release);
    }
    *out = &st;
    return st.status;
}

bool ranges_overlap(uintptr_t a, uint64_t abytes, uintptr_t b, uint64_t bbytes) {
    if (abytes == 0 || bbytes == 0) return false;
    return a < b + bbytes && b < a + abytes;
}

// 2-D tensor map over a rows x cols row-major matrix with row stride ld
// (elements), box box_cols x box_rows, 128-byte swizzle (of 16-byte chunks,
// or of 32-byte chunks for an MN-major TF32 operand), zero fill outside.
int encode_2d(CUtensorMap* map, const void* ptr, int es, int64_t rows, int64_t cols, int64_t ld,
              int box_cols, int box_rows, CUtensorMapDataType dt,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// The 128 x 128-tile FFMA product (with the split or stream-K form the plan
// picks) on B of row stride ldb (b_vec: 16-byte aligned rows).
int ffma_product(const float* A, const float* B, int64_t ldb, bool b_vec, float* C, int64_t M,
                 int64_t K, int64_t N, bool c_vec, const Epilogue& epi, DeviceState* st,
                 cudaStream_t stream) {
    const FfmaPlan plan = ffma_plan((int)M, (int)N, (int)K, st->num_sms);
    void* scratch = nullptr;
    float* partial = nullptr;
    unsigned* counters = nullptr;
    if (plan.split_tiles > 0 && !plan.wide) {
        const int64_t pb = round_up(plan.partial_bytes, 256), cb = round_up(plan.counter_bytes, 256);
        if (cudaMallocFromPoolAsync(&scratch, (size_t)(pb + cb), st->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_NO_MEMORY;
        }
        partial = static_cast<float*>(scratch);
        counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(scratch) + pb);
        // the counters must start at 0 (0.0f has all bits clear)
        if (launch_fill_zero(reinterpret_cast<float*>(counters), cb / 4, stream) != cudaSuccess) {
            cudaFreeAsync(scratch, stream);
            return GEMM_ERR_CUDA;
        }
        g_launches++;
    }
    float* ws = nullptr;
    if (plan.wide) {
        if (cudaMallocFromPoolAsync(&scratch, (size_t)round_up(plan.ws_bytes, 256), st->pool,
                                    stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_NO_MEMORY;
        }
        ws = static_cast<float*>(scratch);
    }
    if (plan.stream) {   // partial tiles, then the per-tile counters (zeroed)
        const int64_t wb = round_up(plan.ws_bytes, 256), cb = round_up(plan.counter_bytes, 256);
        if (cudaMallocFromPoolAsync(&scratch, (size_t)(wb + cb), st->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_NO_MEMORY;
        }
        ws = static_cast<float*>(scratch);
        counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(scratch) + wb);
        if (launch_fill_zero(reinterpret_cast<float*>(counters), cb / 4, stream) != cudaSuccess) {
            cudaFreeAsync(scratch, stream);
            return GEMM_ERR_CUDA;
        }
        g_launches++;
    }
    int rc = GEMM_OK;
    if (launch_ffma_sgemm(A, B, C, (int)M, (int)N, (int)K, (int)ldb, b_vec, c_vec, plan, partial,
                          counters, epi, ws, stream) != cudaSuccess)
        rc = GEMM_ERR_CUDA;
    else
        g_launches++;
    if (rc == GEMM_OK && plan.wide) {
        if (launch_splitk_reduce(ws, plan.splits, M, N, C, M, N, c_vec, epi, st->num_sms, stream) !=
            cudaSuccess)
            rc = GEMM_ERR_CUDA;
        else
            g_launches++;
    }

    if (scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
    return rc;
}

int ffma_gemm(const float* A, const float* B, float* C, int64_t M, int64_t K, int64_t N,
              const Epilogue& epi, DeviceState* st, cudaStream_t stream) {
    const bool b_vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    const bool c_vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
    if (ffma_small_fits(M, N, K, st->num_sms)) {   // small product: 32 x 32 tiles, one launch
        if (launch_ffma_small(A, B, C, (int)M, (int)N, (int)K, b_vec, c_vec, epi, stream) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        g_launches++;
        return GEMM_OK;
    }
    // B rows that are not whole 16-byte chunks would be copied 4 bytes at a
    // time by every tile; with at least kRestrideRows rows of A to amortise
    // it, B is re-strided once into rows padded to 16 bytes (padding zeroed)
    // and read 16 bytes at a time.  (4096 x 4096 x 4090: 2.69 -> 2.26 ms; at
    // M = 256 the copy cost more than it saved.)
    constexpr int64_t kRestrideRows = 1024;
    if (b_vec || M < kRestrideRows)
        return ffma_product(A, B, N, b_vec, C, M, K, N, c_vec, epi, st, stream);
    const int64_t ldb = round_up(N, 4);
    void* b_scratch = nullptr;
    if (cudaMallocFromPoolAsync(&b_scratch, (size_t)round_up(K * ldb * 4, 256), st->pool,
                                stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
    }
    int rc = GEMM_OK;
    if (launch_restride(B, b_scratch, K, N, N, ldb, 4, stream) != cudaSuccess) {
        rc = GEMM_ERR_CUDA;
    } else {
        g_launches++;
        rc = ffma_product(A, static_cast<const float*>(b_scratch), ldb, true, C, M, K, N, c_vec, epi,
                          st, stream);
    }
    if (cudaFreeAsync(b_scratch, stream) != cudaSuccess && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
    return rc;
}

CUtensorMapDataType tensor_type(TcMode mode) {
    return mode == TcMode::kTF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
           : mode == TcMode::kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// The product on operands TMA can read: A (M x K, row stride lda) and B
// (K x N, row stride ldb), 16-byte aligned bases and strides.  With a K
// split (split.splits > 1) the pair kernel computes the whole tiles into C
// and stores the split units' raw partials as 256 x 256 blocks of the
// workspace ws; the reduce kernel then adds each split tile's blocks in
// split order, applies the epilogue and writes C.
int tc_launch(TcMode mode, const void* a_use, int64_t lda, const void* b_use, int64_t ldb,
              float* C, int64_t M, int64_t K, int64_t N, const Epilogue& epi,
              const TcSplit& split, void* ws, DeviceState* st, cudaStream_t stream) {
    const int es = mode == TcMode::kTF32 ? 4 : 2;
    const CUtensorMapDataType dt = tensor_type(mode);
    const TcShape shape = tc_shape(mode);
    // the 2-SM kernel (CTA pairs) when the device can hold pair clusters
    const bool pairs = tc_max_pairs() > 0;
    CUtensorMap map_a, map_b;
    int rc = encode_2d(&map_a, a_use, es, M, K, lda, shape.k_elems, shape.block_m, dt);
    // An MN-major B of 32-bit elements lands in the 128-byte swizzle of
    // 32-byte chunks, the layout kind::tf32 reads such an operand in.
    const CUtensorMapSwizzle b_swizzle =
        es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
    // B in swizzle atoms ordered [k group][column block] (one 4-D box per
    // stage) where the 4-D view covers B exactly, else in 2-D column boxes.
    const bool b_atoms = tc_b_atoms(mode, K, N, ldb);
    if (rc == GEMM_OK && b_atoms) {
        const cuuint64_t dims[4] = {(cuuint64_t)shape.b_box_n, (cuuint64_t)shape.b_atom_rows,
                                    (cuuint64_t)(N / shape.b_box_n),
                                    (cuuint64_t)(K / shape.b_atom_rows)};
        const cuuint64_t strides[3] = {(cuuint64_t)(N * es), (cuuint64_t)(shape.b_box_n * es),
                                       (cuuint64_t)(N * es * shape.b_atom_rows)};
        const cuuint32_t box[4] = {(cuuint32_t)shape.b_box_n, (cuuint32_t)shape.b_atom_rows,
                                   (cuuint32_t)shape.b_blocks,
                                   (cuuint32_t)(shape.k_elems / shape.b_atom_rows)};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        rc = g_encode(&map_b, dt, 4, const_cast<void*>(b_use), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, b_swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
                 ? GEMM_OK
                 : GEMM_ERR_CUDA;
    } else if (rc == GEMM_OK) {
        rc = encode_2d(&map_b, b_use, es, K, N, ldb, shape.b_box_n, shape.k_elems, dt, b_swizzle);
    }
    if (rc != GEMM_OK) return rc;
    const bool c_vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
    // C as a TMA store target (32 x 32 fp32 boxes) when its rows are 16-byte aligned
    CUtensorMap map_c;
    const bool c_tma = pairs && c_vec &&
                       encode_2d(&map_c, C, 4, M, N, N, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) == GEMM_OK;
    const CUtensorMap* mc = c_tma ? &map_c : nullptr;
    if (split.splits > 1) {
        if (!pairs || !ws) return GEMM_ERR_INVALID_ARG;
        const int64_t bytes = tc_split_workspace_bytes(split, M, N);
        CUtensorMap map_w;
        rc = encode_2d(&map_w, ws, 4, bytes / (256 * 4), 256, 256, 32, 32,
                       CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
        if (rc != GEMM_OK) return rc;
        if (launch_tc_gemm_pair(mode, map_a, map_b, mc, &map_w, C, (int)M, (int)N, (int)K, c_vec,
                                epi, split, b_atoms, st->err, kWaitLimitNs, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        g_launches++;
        if (launch_tc_tile_reduce(static_cast<const float*>(ws), split, C, (int)M, (int)N, c_vec,
                                  epi, st->num_sms, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        g_launches++;
        return GEMM_OK;
    }
    const cudaError_t e =
        pairs ? launch_tc_gemm_pair(mode, map_a, map_b, mc, nullptr, C, (int)M, (int)N, (int)K,
                                    c_vec, epi, kNoSplit, b_atoms, st->err, kWaitLimitNs, stream)
              : launch_tc_gemm(mode, map_a, map_b, C, (int)M, (int)N, (int)K, c_vec, epi,
                               st->num_sms, st->err, kWaitLimitNs, stream);
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    g_launches++;
    return GEMM_OK;
}

int tensor_core_gemm(TcMode mode, const void* A, const void* B, float* C, int64_t M, int64_t K,
                     int64_t N, const Epilogue& epi, DeviceState* st, cudaStream_t stream) {
    const TcPlan plan = tc_plan(mode, A, B, M, K, N);
    void* scratch = nullptr;
    if (plan.scratch_bytes() > 0 &&
        cudaMallocFromPoolAsync(&scratch, (size_t)plan.scratch_bytes(), st->pool, stream) !=
            cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
    }
    int rc = tc_product(plan, A, B, C, M, K, N, epi, scratch, stream);
    if (scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
    return rc;
}

// GEMM_FP32_VIA_BF16: round A and B to bfloat16 into scratch rows whose
// stride is a multiple of 16 bytes (TMA-ready), then the BF16 product
// (with the split workspace, when the product is split, after them).
int rounded_bf16_gemm(const float* A, const float* B, float* C, int64_t M, int64_t K, int64_t N,
                      const Epilogue& epi, DeviceState* st, cudaStream_t stream) {
    // A's rows in whole 128-byte lines (no box row straddles two); B's in
    // 16-byte chunks, so that B stays in the atom-ordered form when N allows
    const int64_t lda = round_up(K, 64), ldb = round_up(N, 8);
    const int64_t a_bytes = round_up(M * lda * 2, 256), b_bytes = round_up(K * ldb * 2, 256);
    const TcSplit split = tc_plan_split(TcMode::kBF16, M, N, K);
    const int64_t ws_bytes = round_up(tc_split_workspace_bytes(split, M, N), 256);
    void* scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, (size_t)(a_bytes + b_bytes + ws_bytes), st->pool,
                                stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
    }
    uint8_t* s = static_cast<uint8_t*>(scratch);
    int rc = GEMM_OK, launched = 0;
    if (launch_to_bf16_pair(A, s, M, K, lda, B, s + a_bytes, K, N, ldb, stream, &launched) !=
        cudaSuccess)
        rc = GEMM_ERR_CUDA;
    g_launches += launched;
    if (rc == GEMM_OK)
        rc = tc_launch(TcMode::kBF16, s, lda, s + a_bytes, ldb, C, M, K, N, epi, split,
                       ws_bytes ? s + a_bytes + b_bytes : nullptr, st, stream);
    if (cudaFreeAsync(scratch, stream) != cudaSuccess && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
    return rc;
}

// GEMM_TF32_RN: round A and B to TF32 to nearest (ties away from zero) into
// scratch rows whose stride is a multiple of 16 bytes, then the TF32 product
// (which reads these rounded values exactly; the split workspace, when the
// product is split, after them).
int rounded_tf32_gemm(const float* A, const float* B, float* C, int64_t M, int64_t K, int64_t N,
                      const Epilogue& epi, DeviceState* st, cudaStream_t stream) {
    // A's rows in whole 128-byte lines, B's in 16-byte chunks (as above)
    const int64_t lda = round_up(K, 32), ldb = round_up(N, 4);
    const int64_t a_bytes = round_up(M * lda * 4, 256), b_bytes = round_up(K * ldb * 4, 256);
    const TcSplit split = tc_plan_split(TcMode::kTF32, M, N, K);
    const int64_t ws_bytes = round_up(tc_split_workspace_bytes(split, M, N), 256);
    void* scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, (size_t)(a_bytes + b_bytes + ws_bytes), st->pool,
                                stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
    }
    uint8_t* s = static_cast<uint8_t*>(scratch);
    float* a_r = reinterpret_cast<float*>(s);
    float* b_r = reinterpret_cast<float*>(s + a_bytes);
    int rc = GEMM_OK, launched = 0;
    if (launch_to_tf32_pair(A, a_r, M, K, lda, B, b_r, K, N, ldb, stream, &launched) !=
        cudaSuccess)
        rc = GEMM_ERR_CUDA;
    g_launches += launched;
    if (rc == GEMM_OK)
        rc = tc_launch(TcMode::kTF32, a_r, lda, b_r, ldb, C, M, K, N, epi, split,
                       ws_bytes ? s + a_bytes + b_bytes : nullptr, st, stream);
    if (cudaFreeAsync(scratch, stream) != cudaSuccess && rc == GEMM_OK) rc = GEMM_ERR_CUDA;
    return rc;
}

}  // namespace

// Internal hooks for other translation units of this library (declared in
// kernels.h); they reuse the set-up above without changing it.
namespace libgemm {

int device_setup(int* num_sms, unsigned** err) {
    DeviceState* st = nullptr;
    const int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    *num_sms = st->num_sms;
    *err = st->err;
    return GEMM_OK;
}

TcPlan tc_plan(TcMode mode, const void* A, const void* B, int64_t M, int64_t K, int64_t N) {
    const int es = mode == TcMode::kTF32 ? 4 : 2;
    const int64_t align_elems = 16 / es;
    TcPlan p;
    p.mode = mode;
    // TMA wants 16-byte aligned bases and row strides that are multiples of
    // 16 bytes; an operand that has neither is copied with a padded stride.
    // B is read as the caller stores it (K x N rows, MN-major) in every mode.
    p.pad_a = (K % align_elems) != 0 || (reinterpret_cast<uintptr_t>(A) & 15u) != 0;
    p.pad_b = (N % align_elems) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0;
    // a re-strided operand gets rows of whole 128-byte lines, so that no row
    // of a box straddles two lines (a re-strided B is read in 2-D boxes
    // anyway: the atom-ordered form needs ldb == N)
    p.lda = p.pad_a ? round_up(K, 128 / es) : K;
    p.ldb = p.pad_b ? round_up(N, 128 / es) : N;
    p.a_bytes = p.pad_a ? round_up(M * p.lda * es, 256) : 0;
    p.b_bytes = p.pad_b ? round_up(K * p.ldb * es, 256) : 0;
    p.split = tc_plan_split(mode, M, N, K);
    p.ws_bytes = round_up(tc_split_workspace_bytes(p.split, M, N), 256);
    return p;
}

int tc_product(const TcPlan& plan, const void* A, const void* B, float* C, int64_t M, int64_t K,
               int64_t N, const Epilogue& epi, void* scratch, cudaStream_t stream) {
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    if (plan.scratch_bytes() > 0 && !scratch) return GEMM_ERR_INVALID_ARG;
    const int es = plan.mode == TcMode::kTF32 ? 4 : 2;
    uint8_t* s = static_cast<uint8_t*>(scratch);
    const void* a_use = A;
    const void* b_use = B;
    if (plan.pad_a) {
        if (launch_restride(A, s, M, K, K, plan.lda, es, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        g_launches++;
        a_use = s;
    }
    if (plan.pad_b) {
        if (launch_restride(B, s + plan.a_bytes, K, N, N, plan.ldb, es, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        g_launches++;
        b_use = s + plan.a_bytes;
    }
    void* ws = plan.ws_bytes ? s + plan.a_bytes + plan.b_bytes : nullptr;
    return tc_launch(plan.mode, a_use, plan.lda, b_use, plan.ldb, C, M, K, N, epi, plan.split, ws,
                     st, stream);
}

void count_launch() { g_launches++; }

}  // namespace libgemm

namespace {

// Validation and dispatch shared by gemm() and gemm_ex().
int gemm_impl(const void* A, const void* B, float* C, int64_t M, int64_t K, int64_t N,
              float alpha, float beta, int precision_mode, cudaStream_t stream) {
    if (precision_mode != GEMM_FP32 && precision_mode != GEMM_TF32 && precision_mode != GEMM_BF16 &&
        precision_mode != GEMM_FP16 && precision_mode != GEMM_FP32_VIA_BF16 &&
        precision_mode != GEMM_TF32_RN)
        return GEMM_ERR_INVALID_ARG;
    if (M < 0 || K < 0 || N < 0) return GEMM_ERR_INVALID_ARG;
    // Every dimension must fit the kernels' 32-bit indices and TMA coordinates.
    const int64_t kDimMax = 0x7FFFFFFF;
    if (M > kDimMax || K > kDimMax || N > kDimMax) return GEMM_ERR_INVALID_ARG;
    const int es = (precision_mode == GEMM_BF16 || precision_mode == GEMM_FP16) ? 2 : 4;
    const int64_t kElemMax = INT64_MAX / 16;
    if ((K && M > kElemMax / K) || (N && K > kElemMax / N) || (N && M > kElemMax / N))
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 3u) || (reinterpret_cast<uintptr_t>(A) & (es - 1)) ||
        (reinterpret_cast<uintptr_t>(B) & (es - 1)))
        return GEMM_ERR_MISALIGNED;
    const uint64_t c_bytes = (uint64_t)(M * N) * 4;
    if (K > 0 && (ranges_overlap((uintptr_t)C, c_bytes, (uintptr_t)A, (uint64_t)(M * K) * es) ||
                  ranges_overlap((uintptr_t)C, c_bytes, (uintptr_t)B, (uint64_t)(K * N) * es)))
        return GEMM_ERR_INVALID_ARG;

    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;

    // K == 0 (the empty sum) or alpha == 0: C := beta * C, and A, B are not
    // read; beta == 0 gives 0 without reading C, beta == 1 leaves C as it is.
    if (K == 0 || alpha == 0.0f) {
        if (beta == 1.0f) return GEMM_OK;
        const cudaError_t e = beta == 0.0f ? launch_fill_zero(C, M * N, stream)
                                           : launch_scale(C, M * N, beta, stream);
        if (e != cudaSuccess) return GEMM_ERR_CUDA;
        g_launches++;
        return GEMM_OK;
    }
    const Epilogue epi{alpha, beta, beta != 0.0f ? 2 : (alpha != 1.0f ? 1 : 0)};
    if (precision_mode == GEMM_FP32) return ffma_gemm(static_cast<const float*>(A),
                                                      static_cast<const float*>(B), C, M, K, N, epi,
                                                      st, stream);
    if (precision_mode == GEMM_FP32_VIA_BF16)
        return rounded_bf16_gemm(static_cast<const float*>(A), static_cast<const float*>(B), C, M,
                                 K, N, epi, st, stream);
    if (precision_mode == GEMM_TF32_RN)
        return rounded_tf32_gemm(static_cast<const float*>(A), static_cast<const float*>(B), C, M,
                                 K, N, epi, st, stream);
    const TcMode tm = precision_mode == GEMM_BF16   ? TcMode::kBF16
                      : precision_mode == GEMM_FP16 ? TcMode::kF16
                                                    : TcMode::kTF32;
    return tensor_core_gemm(tm, A, B, C, M, K, N, epi, st, stream);
}

}  // namespace

extern "C" {

int gemm(const void* A, const void* B, float* C, int64_t M, int64_t K, int64_t N,
         int precision_mode, struct CUstream_st* stream) {
    return gemm_impl(A, B, C, M, K, N, 1.0f, 0.0f, precision_mode,
                              reinterpret_cast<cudaStream_t>(stream));
}

int gemm_ex(const void* A, const void* B, float* C, int64_t M, int64_t K, int64_t N, float alpha,
            float beta, int precision_mode, struct CUstream_st* stream) {
    return gemm_impl(A, B, C, M, K, N, alpha, beta, precision_mode,
                              reinterpret_cast<cudaStream_t>(stream));
}

const char* gemm_status_string(int status) {
    switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case GEMM_ERR_CUDA: return "CUDA error";
    case GEMM_ERR_NO_MEMORY: return "scratch allocation failed";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case GEMM_ERR_BOUNDS: return "a kernel access outside its buffer was detected and skipped (debug build)";
    case GEMM_ERR_SCRATCH_LIMIT:
        return "the product needs more scratch than the no-allocation entry point's static buffer";
    default: return "unknown status";
    }
}

int gemm_debug_status(struct CUstream_st* stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, st->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    // debug build: the bounds-check flags of every kernel (read and cleared)
    const unsigned bounds =
        ffma_debug_flags() | ffma_small_debug_flags() | tc_debug_flags() | prep_debug_flags();
    if (word == 0) return bounds ? GEMM_ERR_BOUNDS : GEMM_OK;
    const unsigned zero = 0;
    if (cudaMemcpy(st->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_ERR_TIMEOUT;
}

int gemm_debug_build(void) { return kDebugBuild ? 1 : 0; }

int gemm_version(void) { return 200; }

int64_t gemm_launch_count(void) { return g_launches.load(); }

int gemm_selftest_bounded_wait(int64_t timeout_ns, struct CUstream_st* stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    DeviceState* st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 2000000000) timeout_ns = 2000000000;
    rc = gemm_debug_status(stream_);   // start from a clear error word
    if (rc != GEMM_OK && rc != GEMM_ERR_TIMEOUT) return rc;
    if (launch_wait_selftest(st->err, (uint64_t)timeout_ns, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    g_launches++;
    return gemm_debug_status(stream_);
}

}  // extern "C"
