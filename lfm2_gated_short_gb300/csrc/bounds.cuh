// bounds.cuh -- global-memory bounds checks of the bounds-checked build.
//
// Built with -DSC_BOUNDS_CHECK, every global load and store a kernel makes
// through the helpers below first checks that its whole byte range lies in
// one of the buffers the current call declared (and, for a store, one the
// call may write). A range outside them sets SC_DEV_OUT_OF_BOUNDS in the
// unit's error word, records the first offending address, and is skipped: a
// load returns zeros, a store writes nothing, a bulk copy into shared memory
// is not issued but its bytes are still counted on the mbarrier, so no wait
// is left hanging. Nothing traps.
//
// The table of buffers lives in each translation unit's device memory and is
// filled by the entry point before its launch (bounds_install_here, a
// stream-ordered copy), so calls that overlap on the GPU would share it: the
// checked build is for sequential test runs. Tiled tensor copies (TMA with a
// tensor map) are not checked here: the map's extents bound them in hardware.
//
// In the standard build every check is the constant true and the helpers are
// the plain accesses.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "errors.cuh"
#include "kernels.h"
#include "shortconv.h"

namespace sc {

#ifdef SC_BOUNDS_CHECK

static __device__ BoundsRegion g_bounds_regions[kMaxBoundsRegions];
static __device__ int g_bounds_n;
static __device__ unsigned long long g_bounds_first_bad;  // first address refused, 0 = none

static __device__ __noinline__ bool bounds_ok(const void *p, uint64_t bytes, bool write) {
    const uint64_t a = reinterpret_cast<uint64_t>(p);
    const int n = g_bounds_n < kMaxBoundsRegions ? g_bounds_n : kMaxBoundsRegions;
    for (int i = 0; i < n; ++i) {
        const BoundsRegion r = g_bounds_regions[i];
        if (a >= r.base && bytes <= r.bytes && a - r.base <= r.bytes - bytes &&
            (!write || r.writable))
            return true;
    }
    atomicCAS(&g_bounds_first_bad, 0ull, (unsigned long long)(a | 1ull));
    raise_error(SC_DEV_OUT_OF_BOUNDS);
    return false;
}
#define SC_RD_OK(p, n) ::sc::bounds_ok((p), (uint64_t)(n), false)
#define SC_WR_OK(p, n) ::sc::bounds_ok((p), (uint64_t)(n), true)

// Host side: install this unit's table for the launches that follow on
// `stream` (the copies are stream-ordered; a host copy is kept so a launcher
// can add a buffer of its own, such as a fixed scratch array), and read back
// the first refused address (0 when none) while clearing it.
static BoundsRegion h_bounds_regions[kMaxBoundsRegions];
static int h_bounds_n;

static cudaError_t bounds_install_here(const BoundsRegion *r, int n, cudaStream_t stream) {
    if (n < 0 || n > kMaxBoundsRegions) return cudaErrorInvalidValue;
    for (int i = 0; i < n; ++i) h_bounds_regions[i] = r[i];
    h_bounds_n = n;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_bounds_regions, h_bounds_regions,
                                            sizeof(BoundsRegion) * n, 0,
                                            cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbolAsync(g_bounds_n, &h_bounds_n, sizeof(int), 0,
                                   cudaMemcpyHostToDevice, stream);
}
static cudaError_t bounds_append_here(BoundsRegion r, cudaStream_t stream) {
    if (h_bounds_n >= kMaxBoundsRegions) return cudaErrorInvalidValue;
    BoundsRegion all[kMaxBoundsRegions];
    for (int i = 0; i < h_bounds_n; ++i) all[i] = h_bounds_regions[i];
    all[h_bounds_n] = r;
    return bounds_install_here(all, h_bounds_n + 1, stream);
}
static cudaError_t bounds_take_first_bad_here(cudaStream_t stream, unsigned long long *addr) {
    const unsigned long long zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(addr, g_bounds_first_bad, sizeof(*addr), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_bounds_first_bad, &zero, sizeof(zero), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

#else

#define SC_RD_OK(p, n) true
#define SC_WR_OK(p, n) true

#endif

// A checked scalar or vector load (zeros when refused) and store (skipped).
template <typename V>
__device__ __forceinline__ V gld(const V *p) {
    if (!SC_RD_OK(p, sizeof(V))) return V{};
    return *p;
}
template <typename V>
__device__ __forceinline__ void gst(V *p, const V &v) {
    if (!SC_WR_OK(p, sizeof(V))) return;
    *p = v;
}

}  // namespace sc
