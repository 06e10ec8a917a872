// errors.cuh -- the device error word of one translation unit.
//
// Each .cu file that raises device-side data errors includes this once and
// gets its own word; shortconv_get_error() takes and clears the words of all
// of them. Kernels never trap: they set bits and skip the offending unit.
#pragma once

#include <cuda_runtime.h>

namespace sc {

static __device__ unsigned int g_error_word;   // bit mask of SC_DEV_* codes
static __device__ unsigned int g_error_taken;  // last value taken by take_error_here

static __device__ __forceinline__ void raise_error(unsigned int code) {
    atomicOr(&g_error_word, code);
}

static __global__ void k_take_error() { g_error_taken = atomicExch(&g_error_word, 0u); }

// Take (read and clear) this unit's word, ordered after the stream's work.
static cudaError_t take_error_here(cudaStream_t stream, unsigned int *code) {
    k_take_error<<<1, 1, 0, stream>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbolAsync(code, g_error_taken, sizeof(unsigned int), 0,
                                  cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace sc
