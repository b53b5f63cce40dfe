// noalloc.cu -- gemm_tf32_noalloc: the TF32 tensor-core product with its
// scratch in a static device buffer instead of allocated memory.
//
// Who needs it: callers that cannot allocate device memory at the time they
// multiply -- an application that has reserved the GPU's memory for its own
// pool (an allocation would fail or break its budget), or a latency-critical
// loop that must not stall on, or fail in, an allocator.  gemm() in TF32 mode
// takes its scratch (B^T, and a re-strided A when needed) from the
// stream-ordered allocator; this entry point takes the same scratch from
// g_noalloc_scratch below and calls no allocating routine.
//
// The buffer is a file-scope __device__ array, so each device gets its own
// copy when this library's code is loaded on it.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in object),
// so the first call on a device looks the address up with
// cudaGetSymbolAddress while that device is current, and passes it to the
// kernels.  Calls share the buffer: kernels of overlapping calls race.
#include <cstdint>
#include <mutex>

#include "gemm.h"
#include "kernels.h"

namespace {

using namespace libgemm;

constexpr size_t kScratchBytes = (size_t)GEMM_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // as for gemm(): 2 s per pipeline wait

struct ScratchState {
    bool ready = false;
    void* ptr = nullptr;
};
std::mutex g_mu;
ScratchState g_scratch[kMaxDevices];

// Device address of this device's buffer, looked up once per device.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchState& s = g_scratch[dev];
    if (!s.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        s.ptr = p;
        s.ready = true;
    }
    *out = s.ptr;
    return GEMM_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool overlap(uintptr_t a, uint64_t an, uintptr_t b, uint64_t bn) {
    return an && bn && a < b + bn && b < a + an;
}

}  // namespace

extern "C" int gemm_tf32_noalloc(const float* A, const float* B, float* C, int64_t M, int64_t K,
                                 int64_t N, struct CUstream_st* stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // The same argument rules as gemm().
    if (M < 0 || K < 0 || N < 0) return GEMM_ERR_INVALID_ARG;
    const int64_t kDimMax = 0x7FFFFFFF;
    if (M > kDimMax || K > kDimMax || N > kDimMax) return GEMM_ERR_INVALID_ARG;
    const int64_t kElemMax = INT64_MAX / 16;
    if ((K && M > kElemMax / K) || (N && K > kElemMax / N) || (N && M > kElemMax / N))
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 3u)
        return GEMM_ERR_MISALIGNED;
    const uint64_t c_bytes = (uint64_t)(M * N) * 4;
    if (K > 0 && (overlap((uintptr_t)C, c_bytes, (uintptr_t)A, (uint64_t)(M * K) * 4) ||
                  overlap((uintptr_t)C, c_bytes, (uintptr_t)B, (uint64_t)(K * N) * 4)))
        return GEMM_ERR_INVALID_ARG;

    // Scratch needed: B^T (N x roundup(K, 4)) always, and A re-strided to
    // roundup(K, 4) floats per row when TMA cannot read it in place.
    const bool pad_a = K > 0 && ((K % 4) != 0 || (reinterpret_cast<uintptr_t>(A) & 15u) != 0);
    const int64_t ld = round_up(K, 4);
    const int64_t a_bytes = pad_a ? round_up(M * ld * 4, 256) : 0;
    const int64_t b_bytes = K > 0 ? round_up(N * ld * 4, 256) : 0;
    if ((uint64_t)(a_bytes + b_bytes) > (uint64_t)kScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;

    int num_sms = 0;
    unsigned* err = nullptr;
    int rc = device_setup(&num_sms, &err);
    if (rc != GEMM_OK) return rc;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != GEMM_OK) return rc;

    if (K == 0) {
        if (launch_fill_zero(C, M * N, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        count_launch();
        return GEMM_OK;
    }
    uint8_t* s = static_cast<uint8_t*>(scratch);
    const void* a_use = A;
    if (pad_a) {
        if (launch_restride(A, s, M, K, K, ld, 4, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        count_launch();
        a_use = s;
    }
    void* bt = s + a_bytes;
    if (launch_transpose(B, bt, K, N, ld, 4, num_sms, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    count_launch();

    const TcShape shape = tc_shape(TcMode::kTF32);
    CUtensorMap map_a, map_b;
    rc = encode_tensor_map_2d(&map_a, a_use, 4, M, K, pad_a ? ld : K, shape.k_elems, shape.block_m);
    const bool pairs = tc_max_pairs() > 0;   // the same kernel choice as gemm()
    if (rc == GEMM_OK)
        rc = encode_tensor_map_2d(&map_b, bt, 4, N, K, ld, shape.k_elems,
                                  pairs ? shape.block_n / 2 : shape.block_n);
    if (rc != GEMM_OK) return rc;
    const bool c_vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
    CUtensorMap map_c;
    const bool c_tma =
        pairs && c_vec && encode_tensor_map_2d(&map_c, C, 4, M, N, N, 32, 32) == GEMM_OK;
    const cudaError_t e =
        pairs ? launch_tc_gemm_pair(TcMode::kTF32, true, map_a, map_b, c_tma ? &map_c : nullptr,
                                    nullptr, C, (int)M, (int)N, (int)K, c_vec, kPlainStore, kNoSplit,
                                    err, kWaitLimitNs, stream)
              : launch_tc_gemm(TcMode::kTF32, true, map_a, map_b, C, (int)M, (int)N, (int)K, c_vec,
                               kPlainStore, num_sms, err, kWaitLimitNs, stream);
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    count_launch();
    return GEMM_OK;
}
