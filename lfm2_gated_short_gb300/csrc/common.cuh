// common.cuh -- device helpers shared by the ShortConv kernels.
//
// Every kernel maps one thread to 8 consecutive channels of a row. For bf16
// that is one 128-bit access per array and row (a warp covers 256 channels
// = 512 contiguous bytes); for fp32 it is two 128-bit accesses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sc {

constexpr int kCh = 8;  // channels per thread

// ----------------------------------------------------------- raw 128-bit I/O

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    // Read-only data touched once by this thread: bypass L1, keep L2 default.
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_plain(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void st_plain(void *p, uint4 v) {
    *reinterpret_cast<uint4 *>(p) = v;
}

__device__ __forceinline__ void st_stream(void *p, uint4 v) {
    // Output written once and not re-read by this kernel: evict-first in L2.
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// --------------------------------------------------------- dtype conversion

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even, each half
    return *reinterpret_cast<uint32_t *>(&v);
}

// Storage traits: Q 128-bit words hold the 8 channels of one row section.
template <typename T>
struct Dt;

template <>
struct Dt<__nv_bfloat16> {
    static constexpr int Q = 1;
    // Round an fp32 value to bf16 and back (the value the state stores).
    static __device__ __forceinline__ float round(float v) {
        return __bfloat162float(__float2bfloat16_rn(v));
    }
    static __device__ __forceinline__ void unpack(const uint4 (&q)[Q], float (&f)[kCh]) {
        f[0] = bf16_lo(q[0].x); f[1] = bf16_hi(q[0].x);
        f[2] = bf16_lo(q[0].y); f[3] = bf16_hi(q[0].y);
        f[4] = bf16_lo(q[0].z); f[5] = bf16_hi(q[0].z);
        f[6] = bf16_lo(q[0].w); f[7] = bf16_hi(q[0].w);
    }
    static __device__ __forceinline__ void pack(const float (&f)[kCh], uint4 (&q)[Q]) {
        q[0].x = pack_bf16(f[0], f[1]);
        q[0].y = pack_bf16(f[2], f[3]);
        q[0].z = pack_bf16(f[4], f[5]);
        q[0].w = pack_bf16(f[6], f[7]);
    }
};

template <>
struct Dt<float> {
    static constexpr int Q = 2;
    static __device__ __forceinline__ float round(float v) { return v; }
    static __device__ __forceinline__ void unpack(const uint4 (&q)[Q], float (&f)[kCh]) {
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            f[4 * i + 0] = __uint_as_float(q[i].x);
            f[4 * i + 1] = __uint_as_float(q[i].y);
            f[4 * i + 2] = __uint_as_float(q[i].z);
            f[4 * i + 3] = __uint_as_float(q[i].w);
        }
    }
    static __device__ __forceinline__ void pack(const float (&f)[kCh], uint4 (&q)[Q]) {
#pragma unroll
        for (int i = 0; i < Q; ++i)
            q[i] = make_uint4(__float_as_uint(f[4 * i + 0]), __float_as_uint(f[4 * i + 1]),
                              __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3]));
    }
};

// One row section (8 channels) of an array, as raw words.
template <typename T>
struct Row {
    uint4 q[Dt<T>::Q];
};

template <typename T>
__device__ __forceinline__ Row<T> load_row(const T *p) {
    Row<T> r;
#pragma unroll
    for (int i = 0; i < Dt<T>::Q; ++i) r.q[i] = ld_stream(reinterpret_cast<const uint4 *>(p) + i);
    return r;
}

template <typename T>
__device__ __forceinline__ void store_row(T *p, const float (&f)[kCh]) {
    Row<T> r;
    Dt<T>::pack(f, r.q);
#pragma unroll
    for (int i = 0; i < Dt<T>::Q; ++i) st_stream(reinterpret_cast<uint4 *>(p) + i, r.q[i]);
}

template <typename T>
__device__ __forceinline__ void unpack_row(const Row<T> &r, float (&f)[kCh]) {
    Dt<T>::unpack(r.q, f);
}

// ------------------------------------------- [8 channels][K] blocks (w, state)

// 8*K contiguous elements (channel-major, tap-minor): weights w[h0..h0+7][0..K-1]
// or a state block pool[slot][h0..h0+7][0..K-1]. 8*K*sizeof(T) is a multiple
// of 16 bytes for both dtypes.
template <typename T, int K>
struct Block {
    static constexpr int NQ = kCh * K * (int)sizeof(T) / 16;
};

template <typename T, int K>
__device__ __forceinline__ void load_block(const T *p, float (&f)[kCh][K]) {
    constexpr int NQ = Block<T, K>::NQ;
    uint4 q[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) q[i] = ld_plain(reinterpret_cast<const uint4 *>(p) + i);
    const uint32_t *wd = reinterpret_cast<const uint32_t *>(q);
#pragma unroll
    for (int e = 0; e < kCh * K; ++e) {
        float v;
        if constexpr (sizeof(T) == 2)
            v = (e & 1) ? bf16_hi(wd[e >> 1]) : bf16_lo(wd[e >> 1]);
        else
            v = __uint_as_float(wd[e]);
        f[e / K][e % K] = v;
    }
}

// Values must already be representable in T (the conversion is then exact).
template <typename T, int K>
__device__ __forceinline__ void store_block(T *p, const float (&f)[kCh][K]) {
    constexpr int NQ = Block<T, K>::NQ;
    uint4 q[NQ];
    uint32_t *wd = reinterpret_cast<uint32_t *>(q);
#pragma unroll
    for (int e = 0; e < kCh * K; e += (sizeof(T) == 2 ? 2 : 1)) {
        if constexpr (sizeof(T) == 2)
            wd[e >> 1] = pack_bf16(f[e / K][e % K], f[(e + 1) / K][(e + 1) % K]);
        else
            wd[e] = __float_as_uint(f[e / K][e % K]);
    }
#pragma unroll
    for (int i = 0; i < NQ; ++i) st_plain(reinterpret_cast<uint4 *>(p) + i, q[i]);
}

// ----------------------------------------------------------- the arithmetic

// u = B * x, rounded once to the storage dtype (the value the state keeps).
template <typename T>
__device__ __forceinline__ float gate_in(float b, float x) {
    return Dt<T>::round(__fmul_rn(b, x));
}

// Slide the window by one (oldest out, u in) and return sum_k w_k * win_k.
template <int K>
__device__ __forceinline__ float slide_dot(float (&win)[K], const float (&wk)[K], float u) {
#pragma unroll
    for (int k = 0; k + 1 < K; ++k) win[k] = win[k + 1];
    win[K - 1] = u;
    float z = wk[0] * win[0];
#pragma unroll
    for (int k = 1; k < K; ++k) z = fmaf(wk[k], win[k], z);
    return z;
}

}  // namespace sc
