// common.cuh -- device helpers shared by the ShortConv kernels.
//
// A thread owns a few consecutive channels of a row: 8 in the register-tiled
// prefill (the Row / block helpers below: one 128-bit access per array and
// row in bf16, two in fp32, so a warp covers 512 contiguous bytes), 4 in the
// streamed kernels and decode, 2 in verify (packed pairs and word helpers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"

namespace sc {

constexpr int kCh = 8;  // channels per thread

// Programmatic dependent launch. The kernels are launched with programmatic
// stream serialization, so a kernel may be scheduled while the previous one
// in the stream is still running. pdl_wait() returns once every previous
// kernel has completed and its writes are visible: it comes before a
// kernel's first global memory access. pdl_launch_dependents() lets the next
// kernel be scheduled as soon as this grid's CTAs have all started; that
// kernel still waits for this one to complete before touching memory.
// Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hints that may run before pdl_wait(). prefetch_l2() warms L2 with the line
// holding p and returns nothing to the thread; L2 is the device's point of
// coherence, so an early fetch cannot leave a stale value anywhere a later
// load reads. slot_hint() reads a slot id through L2 only (no L1 line is
// allocated) to choose what to prefetch: before the wait it may be stale, so
// it only ever picks a bounds-checked address and is read again after it.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ int slot_hint(const int32_t *p) {
    if (!SC_RD_OK(p, 4)) return -1;
    return __ldcg(p);
}

// ----------------------------------------------------------- raw 128-bit I/O

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    // Read-only data touched once by this thread: bypass L1, keep L2 default.
    if (!SC_RD_OK(p, 16)) return make_uint4(0u, 0u, 0u, 0u);
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_plain(const void *p) {
    return gld(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_plain(void *p, uint4 v) {
    gst(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ void st_stream(void *p, uint4 v) {
    // Output written once and not re-read by this kernel: evict-first in L2.
    if (!SC_WR_OK(p, 16)) return;
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

// ------------------------------------------------ packed pairs (sm_100 family)
//
// Two fp32 lanes in one 64-bit register (f32x2) and two bf16 lanes in one
// 32-bit register. mul.rn.bf16x2 rounds the exact product once to bf16, the
// same value as gate_in<bf16>; fma.rn.f32x2 / mul.rn.f32x2 round each lane
// exactly like the scalar fmaf / multiply. Kernels using these produce the
// same bits as the scalar helpers above when they keep the operation order.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ f32x2 bf2_to_f2(uint32_t w) {
    return f2_make(bf16_lo(w), bf16_hi(w));
}
__device__ __forceinline__ uint32_t f2_to_bf2(f32x2 v) {
    float lo, hi;
    f2_split(v, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));  // hi -> upper half
    return r;
}

// CPT consecutive channels of one row section (CPT = 2, 4 or 8) as raw
// 32-bit words, loaded from shared memory and stored to global memory with
// one access of CPT * sizeof(T) bytes (two for 32 bytes).
template <typename T, int CPT>
struct Sec {
    static constexpr int NW = CPT * (int)sizeof(T) / 4;  // 32-bit words
    static constexpr int NP = CPT / 2;                    // channel pairs
    uint32_t w[NW];
};

__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t *w, int nw) {
    if (nw == 1) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[0]) : "r"(addr));
    } else if (nw == 2) {
        asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
    } else {
        for (int i = 0; i < nw; i += 4)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[i]), "=r"(w[i + 1]), "=r"(w[i + 2]), "=r"(w[i + 3])
                         : "r"(addr + 4 * i));
    }
}

__device__ __forceinline__ void stg_words(void *p, const uint32_t *w, int nw) {
    if (!SC_WR_OK(p, 4 * nw)) return;
    if (nw == 1) {
        asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(w[0]) : "memory");
    } else if (nw == 2) {
        asm volatile("st.global.cs.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(w[0]), "r"(w[1])
                     : "memory");
    } else {
        for (int i = 0; i < nw; i += 4)
            asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"((char *)p + 4 * i),
                         "r"(w[i]), "r"(w[i + 1]), "r"(w[i + 2]), "r"(w[i + 3])
                         : "memory");
    }
}

template <typename T, int CPT>
__device__ __forceinline__ Sec<T, CPT> lds_sec(uint32_t addr) {
    Sec<T, CPT> r;
    lds_words(addr, r.w, Sec<T, CPT>::NW);
    return r;
}

// u = round(B * x) and widening of C, as CPT/2 f32x2 pairs, and the y store.
template <typename T, int CPT>
struct Pairs;

template <int CPT>
struct Pairs<__nv_bfloat16, CPT> {
    using S = Sec<__nv_bfloat16, CPT>;
    static __device__ __forceinline__ void widen(const S &r, f32x2 (&f)[S::NP]) {
#pragma unroll
        for (int p = 0; p < S::NP; ++p) f[p] = bf2_to_f2(r.w[p]);
    }
    static __device__ __forceinline__ void gate(const S &b, const S &x, f32x2 (&u)[S::NP]) {
#pragma unroll
        for (int p = 0; p < S::NP; ++p) u[p] = bf2_to_f2(bf2_mul(b.w[p], x.w[p]));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *dst, const f32x2 (&y)[S::NP]) {
        uint32_t w[S::NW];
#pragma unroll
        for (int p = 0; p < S::NP; ++p) w[p] = f2_to_bf2(y[p]);
        stg_words(dst, w, S::NW);
    }
};

template <int CPT>
struct Pairs<float, CPT> {
    using S = Sec<float, CPT>;
    static __device__ __forceinline__ void widen(const S &r, f32x2 (&f)[S::NP]) {
#pragma unroll
        for (int p = 0; p < S::NP; ++p)
            f[p] = f2_make(__uint_as_float(r.w[2 * p]), __uint_as_float(r.w[2 * p + 1]));
    }
    static __device__ __forceinline__ void gate(const S &b, const S &x, f32x2 (&u)[S::NP]) {
        f32x2 fb[S::NP], fx[S::NP];
        widen(b, fb);
        widen(x, fx);
#pragma unroll
        for (int p = 0; p < S::NP; ++p) u[p] = f2_mul(fb[p], fx[p]);
    }
    static __device__ __forceinline__ void store(float *dst, const f32x2 (&y)[S::NP]) {
        uint32_t w[S::NW];
#pragma unroll
        for (int p = 0; p < S::NP; ++p) {
            float lo, hi;
            f2_split(y[p], lo, hi);
            w[2 * p] = __float_as_uint(lo);
            w[2 * p + 1] = __float_as_uint(hi);
        }
        stg_words(dst, w, S::NW);
    }
};

// CPT channels x K taps of a [H, K] array (weights or a state), element by
// element (these are read once per sequence, so alignment is not assumed).
template <typename T>
__device__ __forceinline__ float ld_elem(const T *p) {
    if constexpr (sizeof(T) == 2)
        return __uint_as_float((uint32_t)gld(reinterpret_cast<const unsigned short *>(p)) << 16);
    else
        return gld(p);
}
template <typename T>
__device__ __forceinline__ void st_elem(T *p, float v) {  // v representable in T
    if constexpr (sizeof(T) == 2)
        gst(reinterpret_cast<unsigned short *>(p), (unsigned short)(__float_as_uint(v) >> 16));
    else
        gst(p, v);
}
template <typename T, int CPT, int K>
__device__ __forceinline__ void load_taps(const T *p, f32x2 (&f)[K][CPT / 2]) {
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int q = 0; q < CPT / 2; ++q)
            f[k][q] = f2_make(ld_elem(p + (2 * q) * K + k), ld_elem(p + (2 * q + 1) * K + k));
}
template <typename T, int CPT, int K>
__device__ __forceinline__ void store_taps(T *p, const f32x2 (&f)[K][CPT / 2]) {
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int q = 0; q < CPT / 2; ++q) {
            float lo, hi;
            f2_split(f[k][q], lo, hi);
            st_elem(p + (2 * q) * K + k, lo);
            st_elem(p + (2 * q + 1) * K + k, hi);
        }
}

}  // namespace sc
