// debug_checks.cuh -- index checks compiled into the bounds-checked build of libphx.
//
// Built with -DPHX_DEBUG=1 (build.py --debug: _lib/libphx_debug.so), PHX_DCHECK(cond) counts
// every failed condition in a device counter of its translation unit and lets the kernel go
// on: the checks never trap, so a failing check cannot take the GPU down, and the kernel's
// own guards still decide what is read and written.  phx_debug_violations() reads and clears
// the counters.  In the normal build PHX_DCHECK compiles to nothing.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#ifndef PHX_DEBUG
#define PHX_DEBUG 0
#endif

namespace phx {
namespace {

// failed checks in this translation unit since the last read (one counter per unit: the
// library is built without relocatable device code)
__device__ unsigned long long g_debug_violations;

__device__ __forceinline__ void debug_violation() { atomicAdd(&g_debug_violations, 1ull); }

// Read and clear this unit's counter on the current device (-1 if that failed).
inline int64_t debug_take_local() {
    unsigned long long v = 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v) != cudaSuccess ||
        cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return static_cast<int64_t>(v);
}

}  // namespace
}  // namespace phx

#if PHX_DEBUG
#define PHX_DCHECK(cond)                              \
    do {                                              \
        if (!(cond)) ::phx::debug_violation();        \
    } while (0)
#else
#define PHX_DCHECK(cond) \
    do {                 \
    } while (0)
#endif
