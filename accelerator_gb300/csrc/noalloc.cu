// noalloc.cu -- gemm_tf32_noalloc: the TF32 tensor-core product with its
// scratch in a static device buffer instead of allocated memory.
//
// Who needs it: callers that cannot allocate device memory at the time they
// multiply -- an application that has reserved the GPU's memory for its own
// pool (an allocation would fail or break its budget), or a latency-critical
// loop that must not stall on, or fail in, an allocator.  gemm() in TF32 mode
// takes its scratch (re-strided operands, the K-split workspace) from the
// stream-ordered allocator; this entry point plans the product exactly as
// gemm() does (tc_plan: the same kernels, the same K split, so the same
// values bit for bit), takes the same scratch from g_noalloc_scratch below
// and calls no allocating routine.
//
// The buffer is a file-scope __device__ array, so each device gets its own
// copy when this file's device code is loaded on it.  Host code cannot use
// the array's name as a device address (on the host it names a stand-in
// object), so the first call on a device looks the address up with
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

    // Per-device set-up (as gemm() does it), and the buffer's device address:
    // both are done by the first call on a device, whatever it needs.
    int num_sms = 0;
    unsigned* err = nullptr;
    int rc = device_setup(&num_sms, &err);
    if (rc != GEMM_OK) return rc;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != GEMM_OK) return rc;
    if (K == 0) {   // the empty sum: C := 0, nothing read, no scratch
        if (launch_fill_zero(C, M * N, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        count_launch();
        return GEMM_OK;
    }
    // The plan gemm() makes for this product: re-strided A and B when TMA
    // cannot read them in place, and the workspace of a K split.
    const TcPlan plan = tc_plan(TcMode::kTF32, A, B, M, K, N);
    if ((uint64_t)plan.scratch_bytes() > (uint64_t)kScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;
    return tc_product(plan, A, B, C, M, K, N, kPlainStore, scratch, stream);
}
