// debug.cuh -- device-side bounds checks of the debug build.
//
// compute-sanitizer is not available where this library is tested, so the
// debug build (compiled with -DGEMM_DEBUG) checks the global-memory accesses
// of every kernel against the buffer they belong to: an access whose bytes
// do not lie wholly inside [base, base + extent) is skipped and recorded in a
// flag word, and gemm_debug_status() then returns GEMM_ERR_BOUNDS.  Nothing
// traps.  In the release build GEMM_DBG_OK(...) is the constant `true` (its
// arguments are not evaluated), so the kernels compile as if the checks were
// absent.
//
// Each translation unit that includes this header has its own flag word
// (no relocatable device code), and defines a host reader with
// LIBGEMM_DEBUG_READER(name): `unsigned name()` returns that unit's word and
// clears it (always 0 in the release build).
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace libgemm {

#ifdef GEMM_DEBUG
constexpr bool kDebugBuild = true;

namespace dbg {
static __device__ unsigned g_flags;   // one per translation unit

// True when the `bytes` bytes at p lie inside [base, base + extent).
__device__ __forceinline__ bool check(const void* p, const void* base, int64_t extent,
                                      int bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    const bool ok = a >= b && extent >= bytes && a - b <= (uintptr_t)(extent - bytes);
    if (!ok) atomicOr(&g_flags, 1u);
    return ok;
}
}  // namespace dbg

#define GEMM_DBG_OK(p, base, extent, bytes)                                               \
    ::libgemm::dbg::check((const void*)(p), (const void*)(base), (int64_t)(extent), \
                          (int)(bytes))
#define LIBGEMM_DEBUG_READER(name)                                                  \
    unsigned name() {                                                               \
        unsigned v = 0, z = 0;                                                      \
        if (cudaMemcpyFromSymbol(&v, ::libgemm::dbg::g_flags, sizeof v) != cudaSuccess) \
            return cudaGetLastError(), 0u;                                          \
        cudaMemcpyToSymbol(::libgemm::dbg::g_flags, &z, sizeof z);                  \
        return v;                                                                   \
    }
#else
constexpr bool kDebugBuild = false;
#define GEMM_DBG_OK(p, base, extent, bytes) true
#define LIBGEMM_DEBUG_READER(name) \
    unsigned name() { return 0u; }
#endif

}  // namespace libgemm
