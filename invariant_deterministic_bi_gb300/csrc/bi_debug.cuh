// bi_debug.cuh -- bounds checks of the debug build (libbi_debug.so).
//
// In a translation unit compiled with -DBI_DEBUG=1, BI_IN_BOUNDS(cond, status)
// evaluates cond; when it is false it records kDevBounds in the device status
// word, with the source line of the first failing check in the word's upper
// 16 bits, and yields false, so that the caller skips the access it guards.
// It never traps, asserts or stops the kernel. In the release build it is the
// constant true and compiles away. compute-sanitizer is closed on the GPUs this
// library is tested on; these checks stand in for its bounds checking.
#pragma once
#include <cstdint>

namespace bi {

constexpr unsigned kDevBounds = 4u;       // a debug-build bounds check failed (the access was skipped)

#ifdef BI_DEBUG
__device__ __forceinline__ bool bounds_check(bool ok, unsigned *status, unsigned line) {
    if (!ok && status) {
        const unsigned old = atomicOr(status, kDevBounds);
        if ((old >> 16) == 0) atomicCAS(status, old | kDevBounds, old | kDevBounds | ((line & 0xFFFFu) << 16));
    }
    return ok;
}
#define BI_IN_BOUNDS(cond, status) (::bi::bounds_check((cond), (status), __LINE__))
constexpr bool kDebugBuild = true;
#else
#define BI_IN_BOUNDS(cond, status) true
constexpr bool kDebugBuild = false;
#endif

}  // namespace bi
