// forward.cu -- ShortConv forward kernels: varlen prefill, decode, speculative
// verify and rollback.
//
// The arithmetic is the MAX LFM2ShortConv definition ("MAX Pipelines 的 LFM2
// 架构支持", section "短卷积实现（LFM2ShortConv）"): u = B*x (rounded to the
// storage dtype, the value the state keeps), a K-wide window sliding by one
// per token, z = sum_k w_k window_k in fp32, y = C*z rounded once.
//
// Instead of the page's sequential per-token loop, prefill is a parallel FIR:
// each thread owns 8 channels and a tile of L consecutive rows and rebuilds
// the K-1 values of u before its tile from the B and x rows just above it.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "errors.cuh"
#include "kernels.h"
#include "launch.h"
#include "shortconv.h"
#include "tma.cuh"

namespace sc {

constexpr int kThreads = 256;
constexpr int kMaxStagedSeqs = 2048;  // cu_seqlens entries staged in shared memory
constexpr int kChunk = 4;             // rows whose loads are issued together

// u of one row (8 channels) from its B and x sections.
template <typename T>
__device__ __forceinline__ void row_u(const T *__restrict__ bcx, int64_t row, int H, int h0,
                                      float (&u)[kCh]) {
    const T *p = bcx + row * 3 * (int64_t)H + h0;
    const Row<T> rb = load_row(p), rx = load_row(p + 2 * H);
    float b[kCh], x[kCh];
    unpack_row(rb, b);
    unpack_row(rx, x);
#pragma unroll
    for (int c = 0; c < kCh; ++c) u[c] = gate_in<T>(b[c], x[c]);
}

// The optional per-channel conv bias of 8 channels (zeros when absent).
template <typename T>
__device__ __forceinline__ void load_bias8(const T *__restrict__ bias, int h0, float (&bh)[kCh]) {
    if (bias != nullptr) {
        unpack_row(load_row(bias + h0), bh);
    } else {
#pragma unroll
        for (int c = 0; c < kCh; ++c) bh[c] = 0.f;
    }
}

// Rows [a, e) of one sequence for 8 channels; `win` enters holding the last K
// values of u before row a and leaves holding the last K up to row e-1.
template <typename T, int K>
__device__ __forceinline__ void run_rows(const T *__restrict__ bcx, int H, int h0, int64_t a,
                                         int64_t e, const float (&wt)[kCh][K],
                                         const float (&bh)[kCh], bool has_bias,
                                         float (&win)[kCh][K], T *__restrict__ y) {
    const int64_t ld = 3 * (int64_t)H;
    for (int64_t r = a; r < e; r += kChunk) {
        Row<T> rb[kChunk], rc[kChunk], rx[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (r + j < e) {
                const T *p = bcx + (r + j) * ld + h0;
                rb[j] = load_row(p);
                rc[j] = load_row(p + H);
                rx[j] = load_row(p + 2 * H);
            }
        }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (r + j < e) {
                float b[kCh], c[kCh], x[kCh], out[kCh];
                unpack_row(rb[j], b);
                unpack_row(rc[j], c);
                unpack_row(rx[j], x);
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) {
                    const float u = gate_in<T>(b[ch], x[ch]);
                    float z = slide_dot<K>(win[ch], wt[ch], u);
                    if (has_bias) z = z + bh[ch];
                    out[ch] = c[ch] * z;
                }
                store_row(y + (r + j) * (int64_t)H + h0, out);
            }
        }
    }
}

#include "prefill_stream.cuh"

// ------------------------------------------------------------ tiled prefill
//
// Unit = (row tile of L rows, channel group cg of 8 channels). A tile may
// hold pieces of several sequences; each piece restarts its window.
//
// Race-free state update: the piece that holds a sequence's FIRST row (its
// "owner") is the only reader of the old slot state, and it is extended to
// cover at least the sequence's first K-1 rows (other tiles start that
// sequence at row s0+K-1 or later, so their history comes from B and x rows
// of the same sequence). The owner also writes the final state, after its own
// read, rebuilding the last K values of u from the sequence's last K rows
// when the sequence ends in another tile.
template <typename T, int K, int L>
__global__ void __launch_bounds__(kThreads)
    k_prefill(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
              const T *__restrict__ bias, const int32_t *__restrict__ cu, int N,
              const int32_t *__restrict__ slots, T *__restrict__ pool, int n_slots,
              T *__restrict__ y) {
    __shared__ int32_t s_cu[kMaxStagedSeqs + 1];
    const bool staged = N <= kMaxStagedSeqs;
    pdl_wait();
    pdl_launch_dependents();

    // The whole call is skipped unless cu_seqlens is 0 = c0 <= ... <= cN = T.
    int bad = 0;
    for (int j = threadIdx.x; j <= N; j += blockDim.x) {
        const int32_t c = gld(cu + j);
        if (staged) s_cu[j] = c;
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && gld(cu + j + 1) < c) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(SC_DEV_BAD_SEQLENS);
        return;
    }

    const int groups = H / kCh;
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n_tiles = (T_rows + L - 1) / L;
    if (unit >= n_tiles * groups) return;
    const int cg = (int)(unit % groups);
    const int h0 = cg * kCh;
    const int64_t r0 = (unit / groups) * L;
    const int64_t r1 = min(r0 + (int64_t)L, T_rows);
    auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : gld(cu + j); };

    // Largest i with cu[i] <= r0: the sequence holding row r0.
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (CU(mid) <= r0) lo = mid; else hi = mid - 1;
    }

    float wt[kCh][K], bh[kCh];
    load_block<T, K>(w + (int64_t)h0 * K, wt);
    load_bias8<T>(bias, h0, bh);
    const bool has_bias = bias != nullptr;

    for (int i = lo; i < N; ++i) {
        const int64_t s0 = CU(i), s1 = CU(i + 1);
        if (s0 >= r1) break;
        if (s1 <= s0) continue;  // empty: its slot keeps its state
        const bool owner = s0 >= r0;
        int64_t a, e;
        if (owner) {
            a = s0;
            e = min(s1, max(r1, s0 + (K - 1)));
        } else {
            a = max(r0, s0 + (K - 1));
            e = min(s1, r1);
            if (a >= e) continue;
        }
        const int slot = gld(slots + i);
        if (slot < 0 || slot >= n_slots) {
            if (owner && cg == 0) raise_error(SC_DEV_BAD_SLOT);
            continue;
        }
        T *st = pool + ((int64_t)slot * H + h0) * K;
        float win[kCh][K];
        if (owner) {
            load_block<T, K>(st, win);
        } else {
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch) win[ch][0] = 0.f;
#pragma unroll
            for (int k = 1; k < K; ++k) {
                float u[kCh];
                row_u<T>(bcx, a - K + k, H, h0, u);
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) win[ch][k] = u[ch];
            }
        }
        run_rows<T, K>(bcx, H, h0, a, e, wt, bh, has_bias, win, y);
        if (owner) {
            if (e < s1) {  // the sequence ends in a later tile: rebuild its last K values
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    float u[kCh];
                    row_u<T>(bcx, s1 - K + k, H, h0, u);
#pragma unroll
                    for (int ch = 0; ch < kCh; ++ch) win[ch][k] = u[ch];
                }
            }
            store_block<T, K>(st, win);
        }
    }
}

template <typename T, int K, int L>
static cudaError_t prefill_inst(const void *bcx, int64_t rows, int H, const void *w,
                                const void *bias, const int32_t *cu, int N,
                                const int32_t *slots, void *pool, int n_slots, void *y,
                                cudaStream_t stream) {
    const int64_t units = (rows + L - 1) / L * (H / kCh);
    int64_t blocks = (units + kThreads - 1) / kThreads;
    if (blocks < 1) blocks = 1;  // still validates cu_seqlens
    return launch_pdl(k_prefill<T, K, L>, dim3((unsigned)blocks), dim3(kThreads), 0, stream,
                      (const T *)bcx, rows, H, (const T *)w, (const T *)bias, cu, N, slots,
                      (T *)pool, n_slots, (T *)y);
}

template <typename T, int K>
static cudaError_t prefill_L(int L, const void *bcx, int64_t rows, int H, const void *w,
                             const void *bias, const int32_t *cu, int N, const int32_t *slots,
                             void *pool, int n_slots, void *y, cudaStream_t s) {
    switch (L) {
        case 4: return prefill_inst<T, K, 4>(bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        case 8: return prefill_inst<T, K, 8>(bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        case 16: return prefill_inst<T, K, 16>(bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        default: return prefill_inst<T, K, 32>(bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
    }
}

template <typename T>
static cudaError_t prefill_K(int K, int L, const void *bcx, int64_t rows, int H, const void *w,
                             const void *bias, const int32_t *cu, int N, const int32_t *slots,
                             void *pool, int n_slots, void *y, cudaStream_t s) {
    switch (K) {
        case 1: return prefill_L<T, 1>(L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        case 2: return prefill_L<T, 2>(L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        case 3: return prefill_L<T, 3>(L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
        default: return prefill_L<T, 4>(L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
    }
}

template <typename T, int K, bool HB>
static cudaError_t prefill_stream_inst(const void *bcx, int64_t rows, int H, const void *w,
                                       const void *bias, const int32_t *cu, int N,
                                       const int32_t *slots, void *pool, int n_slots, void *y,
                                       int sm_count, cudaStream_t stream) {
    const int CW = std::min(kStreamSlice, H);
    const int n_slices = (H + kStreamSlice - 1) / kStreamSlice;
    const int threads = (CW / kStreamCpt + 31) / 32 * 32 + 32;  // consumers + one producer warp
    const size_t smem = stream_smem_bytes<T>(CW);
    auto kern = k_prefill_stream<T, K, HB>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // Opt in to the large dynamic shared memory once per device; remember the
    // occupancy of the last (device, slice width) seen.
    static std::atomic<unsigned long long> configured{0};
    static std::atomic<int> last_key{-1}, last_occ{0};
    if (dev < 64 && !(configured.load() & (1ull << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)stream_smem_bytes<T>(kStreamSlice));
        if (e != cudaSuccess) return e;
        configured.fetch_or(1ull << dev);
    }
    const int key = dev * 4096 + CW / kCh;
    int occ = last_key.load() == key ? last_occ.load() : 0;
    if (occ <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
        if (e != cudaSuccess) return e;
        if (occ <= 0) return cudaErrorInvalidConfiguration;
        last_occ.store(occ);
        last_key.store(key);
    }
    int64_t n_row = std::min<int64_t>((rows + kStreamMinRows - 1) / kStreamMinRows,
                                      (int64_t)sm_count * occ / n_slices);
    if (n_row < 1) n_row = 1;
    return launch_pdl(kern, dim3((unsigned)(n_row * n_slices)), dim3(threads), smem, stream,
                      (const T *)bcx, rows, H, (const T *)w, (const T *)bias, cu, N, slots,
                      (T *)pool, n_slots, (T *)y, n_slices, (int)n_row);
}

template <typename T>
static cudaError_t prefill_stream_K(int K, const void *bcx, int64_t rows, int H, const void *w,
                                    const void *bias, const int32_t *cu, int N,
                                    const int32_t *slots, void *pool, int n_slots, void *y,
                                    int sms, cudaStream_t s) {
#define SC_STREAM_ARGS bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, sms, s
#define SC_STREAM_CASE(k)                                                   \
    return bias != nullptr ? prefill_stream_inst<T, k, true>(SC_STREAM_ARGS) \
                           : prefill_stream_inst<T, k, false>(SC_STREAM_ARGS)
    switch (K) {
        case 1: SC_STREAM_CASE(1);
        case 2: SC_STREAM_CASE(2);
        case 3: SC_STREAM_CASE(3);
        default: SC_STREAM_CASE(4);
    }
#undef SC_STREAM_CASE
#undef SC_STREAM_ARGS
}

cudaError_t launch_prefill(int dtype, int H, int K, const void *bcx, int64_t rows, const void *w,
                           const void *bias, const int32_t *cu, int N, const int32_t *slots,
                           void *pool, int n_slots, void *y, int L, int sm_count,
                           cudaStream_t s) {
    if (L == 0) {
        if (dtype == SC_BF16)
            return prefill_stream_K<__nv_bfloat16>(K, bcx, rows, H, w, bias, cu, N, slots, pool,
                                                   n_slots, y, sm_count, s);
        return prefill_stream_K<float>(K, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y,
                                       sm_count, s);
    }
    if (dtype == SC_BF16)
        return prefill_K<__nv_bfloat16>(K, L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots,
                                        y, s);
    return prefill_K<float>(K, L, bcx, rows, H, w, bias, cu, N, slots, pool, n_slots, y, s);
}

// NW consecutive 32-bit words at p with A-byte accesses (p aligned to A).
template <int NW, int A>
__device__ __forceinline__ void ld_words(const void *p, uint32_t (&w)[NW]) {
    static_assert((NW * 4) % A == 0, "whole accesses");
    if (!SC_RD_OK(p, NW * 4)) {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = 0u;
        return;
    }
#pragma unroll
    for (int i = 0; i < NW * 4 / A; ++i) {
        if constexpr (A == 16) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        } else if constexpr (A == 8) {
            const uint2 v = reinterpret_cast<const uint2 *>(p)[i];
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        } else {
            w[i] = reinterpret_cast<const uint32_t *>(p)[i];
        }
    }
}
template <int NW, int A>
__device__ __forceinline__ void st_words(void *p, const uint32_t (&w)[NW]) {
    if (!SC_WR_OK(p, NW * 4)) return;
#pragma unroll
    for (int i = 0; i < NW * 4 / A; ++i) {
        if constexpr (A == 16)
            reinterpret_cast<uint4 *>(p)[i] =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        else if constexpr (A == 8)
            reinterpret_cast<uint2 *>(p)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
        else
            reinterpret_cast<uint32_t *>(p)[i] = w[i];
    }
}
// Element e of raw words holding T values, as fp32; and the reverse (the value
// is rounded to T, exactly when it is already representable).
template <typename T, int NW>
__device__ __forceinline__ float word_elem(const uint32_t (&w)[NW], int e) {
    if constexpr (sizeof(T) == 2)
        return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else
        return __uint_as_float(w[e]);
}
template <typename T, int NE, int NW>
__device__ __forceinline__ void pack_words(const float (&v)[NE], uint32_t (&w)[NW]) {
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int m = 0; m < NW; ++m) w[m] = pack_bf16(v[2 * m], v[2 * m + 1]);
    } else {
#pragma unroll
        for (int m = 0; m < NW; ++m) w[m] = __float_as_uint(v[m]);
    }
}

// ------------------------------------------------------------------- decode
//
#ifndef SC_DECODE_THREADS
#define SC_DECODE_THREADS 256  // threads per CTA (build-time knob)
#endif
constexpr int kDecodeThreads = SC_DECODE_THREADS;
//
// Unit = (sequence i, CH channels). The token's B, C, x loads do not depend
// on the slot id, so they are issued before the slot-dependent state load.
// CH = 4 by default: at 256 sequences both 8 channels a thread (fewer
// threads to hide the two round trips) and 2 measured slower.
template <typename T, int K, int CH>
__global__ void __launch_bounds__(kDecodeThreads)
    k_decode(const T *__restrict__ bcx, int N, int H, const T *__restrict__ w,
             const T *__restrict__ bias, const int32_t *__restrict__ slots,
             T *__restrict__ pool, int n_slots, T *__restrict__ y) {
    constexpr int NWR = CH * (int)sizeof(T) / 4;
    constexpr int AR = NWR * 4 >= 16 ? 16 : NWR * 4;
    constexpr int SB = CH * K * (int)sizeof(T);
    constexpr int NWS = SB / 4;
    constexpr int AS = SB % 16 == 0 ? 16 : (SB % 8 == 0 ? 8 : 4);
    const int groups = H / CH;
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = unit < (int64_t)N * groups;
    const int i = (int)(unit / groups), cg = (int)(unit % groups), h0 = cg * CH;
    if (live) {  // warm L2 with the slot's state while earlier kernels finish
        const int hint = slot_hint(slots + i);
        if (hint >= 0 && hint < n_slots) prefetch_l2(pool + ((int64_t)hint * H + h0) * K);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (!live) return;
    const T *p = bcx + (int64_t)i * 3 * H + h0;
    uint32_t rb[NWR], rc[NWR], rx[NWR], ww[NWS], sw[NWS], bw[NWR];
    ld_words<NWR, AR>(p, rb);
    ld_words<NWR, AR>(p + H, rc);
    ld_words<NWR, AR>(p + 2 * H, rx);
    const int slot = gld(slots + i);
    ld_words<NWS, AS>(w + (int64_t)h0 * K, ww);
    if (bias != nullptr) ld_words<NWR, AR>(bias + h0, bw);
    if (slot < 0 || slot >= n_slots) {
        if (cg == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    T *st = pool + ((int64_t)slot * H + h0) * K;
    ld_words<NWS, AS>(st, sw);
    float out[CH], nst[CH * K];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        float win[K], wt[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            win[k] = word_elem<T>(sw, c * K + k);
            wt[k] = word_elem<T>(ww, c * K + k);
        }
        float z = slide_dot<K>(win, wt, gate_in<T>(word_elem<T>(rb, c), word_elem<T>(rx, c)));
        if (bias != nullptr) z = z + word_elem<T>(bw, c);
        out[c] = word_elem<T>(rc, c) * z;
#pragma unroll
        for (int k = 0; k < K; ++k) nst[c * K + k] = win[k];
    }
    uint32_t yw[NWR], stw[NWS];
    pack_words<T>(out, yw);
    pack_words<T>(nst, stw);
    st_words<NWR, AR>(y + (int64_t)i * H + h0, yw);
    st_words<NWS, AS>(st, stw);
}

#ifndef SC_DECODE_CH
#define SC_DECODE_CH 4  // channels per decode thread: 2, 4 or 8
#endif

template <typename T, int K>
static cudaError_t decode_inst(const void *bcx, int N, int H, const void *w, const void *bias,
                               const int32_t *slots, void *pool, int n_slots, void *y,
                               cudaStream_t stream) {
    constexpr int CH = SC_DECODE_CH;
    static_assert(CH == 2 || CH == 4 || CH == 8, "H is a multiple of 8");
    const int64_t units = (int64_t)N * (H / CH);
    const int64_t blocks = (units + kDecodeThreads - 1) / kDecodeThreads;
    return launch_pdl(k_decode<T, K, CH>, dim3((unsigned)blocks), dim3(kDecodeThreads), 0,
                      stream, (const T *)bcx, N, H, (const T *)w, (const T *)bias, slots,
                      (T *)pool, n_slots, (T *)y);
}

template <typename T>
static cudaError_t decode_K(int K, const void *bcx, int N, int H, const void *w,
                            const void *bias, const int32_t *slots, void *pool, int n_slots,
                            void *y, cudaStream_t s) {
    switch (K) {
        case 1: return decode_inst<T, 1>(bcx, N, H, w, bias, slots, pool, n_slots, y, s);
        case 2: return decode_inst<T, 2>(bcx, N, H, w, bias, slots, pool, n_slots, y, s);
        case 3: return decode_inst<T, 3>(bcx, N, H, w, bias, slots, pool, n_slots, y, s);
        default: return decode_inst<T, 4>(bcx, N, H, w, bias, slots, pool, n_slots, y, s);
    }
}

cudaError_t launch_decode(int dtype, int H, int K, const void *bcx, int N, const void *w,
                          const void *bias, const int32_t *slots, void *pool, int n_slots,
                          void *y, cudaStream_t s) {
    if (dtype == SC_BF16)
        return decode_K<__nv_bfloat16>(K, bcx, N, H, w, bias, slots, pool, n_slots, y, s);
    return decode_K<float>(K, bcx, N, H, w, bias, slots, pool, n_slots, y, s);
}

// ------------------------------------------------------------------- verify
//
// Unit = (sequence i, CH channels); the D draft steps run in order in
// registers. All draft rows (up to VerifyRows<T> at a time) are requested
// before the slot-dependent state load, so a sequence costs two dependent
// memory round trips. Small CTAs spread the few units over all SMs. CH = 2
// channels a thread by default: at 64 sequences, 8 channels a thread leave
// a few warps per SM, each with a long chain of dependent steps.
#ifndef SC_VERIFY_THREADS
#define SC_VERIFY_THREADS 64  // threads per verify CTA (build-time knob)
#endif
constexpr int kVerifyThreads = SC_VERIFY_THREADS;
// Draft rows held in registers at once: 8 for bf16; 4 for fp32, whose rows
// take twice the registers (8 spilled).
template <typename T>
constexpr int VerifyRows = sizeof(T) == 2 ? 8 : 4;

template <typename T, int K, int CH>
__global__ void __launch_bounds__(kVerifyThreads)
    k_verify(const T *__restrict__ bcx, int N, int D, int H, const T *__restrict__ w,
             const T *__restrict__ bias, const int32_t *__restrict__ slots,
             const T *__restrict__ pool, int n_slots, T *__restrict__ win_out,
             T *__restrict__ y) {
    constexpr int NWR = CH * (int)sizeof(T) / 4;          // words of a row section
    constexpr int AR = NWR * 4 >= 16 ? 16 : NWR * 4;
    constexpr int SB = CH * K * (int)sizeof(T);           // bytes of a [CH][K] block
    constexpr int NWS = SB / 4;
    constexpr int AS = SB % 16 == 0 ? 16 : (SB % 8 == 0 ? 8 : 4);
    constexpr int VR = VerifyRows<T>;
    const int groups = H / CH;
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = unit < (int64_t)N * groups;
    const int i = (int)(unit / groups), cg = (int)(unit % groups), h0 = cg * CH;
    if (live) {  // warm L2 with the slot's state while earlier kernels finish
        const int hint = slot_hint(slots + i);
        if (hint >= 0 && hint < n_slots) prefetch_l2(pool + ((int64_t)hint * H + h0) * K);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (!live) return;
    const int64_t ld = 3 * (int64_t)H;
    const int slot = gld(slots + i);
    uint32_t rb[VR][NWR], rc[VR][NWR], rx[VR][NWR];
    auto load_rows = [&](int j0) {
#pragma unroll
        for (int jj = 0; jj < VR; ++jj) {
            if (j0 + jj < D) {
                const T *p = bcx + ((int64_t)i * D + j0 + jj) * ld + h0;
                ld_words<NWR, AR>(p, rb[jj]);
                ld_words<NWR, AR>(p + H, rc[jj]);
                ld_words<NWR, AR>(p + 2 * H, rx[jj]);
            }
        }
    };
    load_rows(0);
    uint32_t ww[NWS], sw[NWS], bw[NWR];
    ld_words<NWS, AS>(w + (int64_t)h0 * K, ww);
    if (bias != nullptr) ld_words<NWR, AR>(bias + h0, bw);
    if (slot < 0 || slot >= n_slots) {
        if (cg == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    ld_words<NWS, AS>(pool + ((int64_t)slot * H + h0) * K, sw);
    float wt[CH][K], win[CH][K], bh[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        bh[c] = bias != nullptr ? word_elem<T>(bw, c) : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            wt[c][k] = word_elem<T>(ww, c * K + k);
            win[c][k] = word_elem<T>(sw, c * K + k);
        }
    }
    for (int j0 = 0; j0 < D; j0 += VR) {
        if (j0 > 0) load_rows(j0);
#pragma unroll
        for (int jj = 0; jj < VR; ++jj) {
            if (j0 + jj < D) {
                const int64_t t = (int64_t)i * D + j0 + jj;
                float out[CH], st[CH * K];
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const float u = gate_in<T>(word_elem<T>(rb[jj], c), word_elem<T>(rx[jj], c));
                    float z = slide_dot<K>(win[c], wt[c], u);
                    if (bias != nullptr) z = z + bh[c];
                    out[c] = word_elem<T>(rc[jj], c) * z;
#pragma unroll
                    for (int k = 0; k < K; ++k) st[c * K + k] = win[c][k];
                }
                uint32_t yw[NWR], stw[NWS];
                pack_words<T>(out, yw);
                pack_words<T>(st, stw);
                st_words<NWR, AR>(y + t * H + h0, yw);
                st_words<NWS, AS>(win_out + (t * H + h0) * K, stw);
            }
        }
    }
}

#ifndef SC_VERIFY_CH
#define SC_VERIFY_CH 2  // channels per verify thread: 2, 4 or 8
#endif

template <typename T, int K>
static cudaError_t verify_inst(const void *bcx, int N, int D, int H, const void *w,
                               const void *bias, const int32_t *slots, const void *pool,
                               int n_slots, void *win, void *y, cudaStream_t stream) {
    constexpr int CH = SC_VERIFY_CH;
    static_assert(CH == 2 || CH == 4 || CH == 8, "H is a multiple of 8");
    const int64_t units = (int64_t)N * (H / CH);
    const int64_t blocks = (units + kVerifyThreads - 1) / kVerifyThreads;
    return launch_pdl(k_verify<T, K, CH>, dim3((unsigned)blocks), dim3(kVerifyThreads), 0,
                      stream, (const T *)bcx, N, D, H, (const T *)w, (const T *)bias, slots,
                      (const T *)pool, n_slots, (T *)win, (T *)y);
}

template <typename T>
static cudaError_t verify_K(int K, const void *bcx, int N, int D, int H, const void *w,
                            const void *bias, const int32_t *slots, const void *pool,
                            int n_slots, void *win, void *y, cudaStream_t s) {
    switch (K) {
        case 1: return verify_inst<T, 1>(bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
        case 2: return verify_inst<T, 2>(bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
        case 3: return verify_inst<T, 3>(bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
        default: return verify_inst<T, 4>(bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
    }
}

cudaError_t launch_verify(int dtype, int H, int K, const void *bcx, int N, int D, const void *w,
                          const void *bias, const int32_t *slots, const void *pool, int n_slots,
                          void *win, void *y, cudaStream_t s) {
    if (dtype == SC_BF16)
        return verify_K<__nv_bfloat16>(K, bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
    return verify_K<float>(K, bcx, N, D, H, w, bias, slots, pool, n_slots, win, y, s);
}

// ----------------------------------------------------------------- rollback
//
// A plain 16-byte copy of the accepted window record into the slot, for L
// layers at once: layer l's tape is win + l N D (H K) and its pool
// pool + l n_slots (H K); every layer takes the same accepted lengths.
__global__ void __launch_bounds__(kThreads)
    k_rollback(int L, int N, int D, int64_t q_per_seq, const uint4 *__restrict__ win,
               const int32_t *__restrict__ accepted, const int32_t *__restrict__ slots,
               uint4 *__restrict__ pool, int n_slots) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t per_layer = (int64_t)N * q_per_seq;
    if (unit >= (int64_t)L * per_layer) return;
    const int64_t l = unit / per_layer, rem = unit % per_layer;
    const int i = (int)(rem / q_per_seq);
    const int64_t q = rem % q_per_seq;
    const int a = gld(accepted + i), slot = gld(slots + i);
    if (a < 0 || a > D) {
        if (q == 0 && l == 0) raise_error(SC_DEV_BAD_ACCEPTED);
        return;
    }
    if (slot < 0 || slot >= n_slots) {
        if (q == 0 && l == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    if (a == 0) return;
    gst(pool + (l * n_slots + slot) * q_per_seq + q,
        gld(win + ((l * N + i) * D + (a - 1)) * q_per_seq + q));
}

cudaError_t launch_rollback(int dtype, int H, int K, int L, int N, int D, const void *win,
                            const int32_t *accepted, const int32_t *slots, void *pool,
                            int n_slots, cudaStream_t stream) {
    const int64_t elem = dtype == SC_BF16 ? 2 : 4;
    const int64_t q_per_seq = (int64_t)H * K * elem / 16;
    const int64_t blocks = ((int64_t)L * N * q_per_seq + kThreads - 1) / kThreads;
    return launch_pdl(k_rollback, dim3((unsigned)blocks), dim3(kThreads), 0, stream, L, N, D,
                      q_per_seq, (const uint4 *)win, accepted, slots, (uint4 *)pool, n_slots);
}

// ------------------------------------------------------------ error word

cudaError_t read_and_clear_error(cudaStream_t stream, unsigned int *code) {
    unsigned int a = 0, b = 0, c = 0, d = 0;  // forward, backward, slot-pool, projection words
    cudaError_t e = take_error_here(stream, &a);
    if (e != cudaSuccess) return e;
    e = take_error_backward(stream, &b);
    if (e != cudaSuccess) return e;
    e = take_error_slots(stream, &c);
    if (e != cudaSuccess) return e;
    e = take_error_proj(stream, &d);
    if (e != cudaSuccess) return e;
    *code = a | b | c | d;
    return cudaSuccess;
}

#ifdef SC_BOUNDS_CHECK
// ------------------------------------------------- bounds-checked build only

cudaError_t bounds_install(int unit, const BoundsRegion *r, int n, cudaStream_t s) {
    switch (unit) {
        case kUnitForward: return bounds_install_here(r, n, s);
        case kUnitBackward: return bounds_install_backward(r, n, s);
        case kUnitProj: return bounds_install_proj(r, n, s);
        default: return bounds_install_slots(r, n, s);
    }
}

cudaError_t bounds_take_first_bad(cudaStream_t s, unsigned long long *addr) {
    unsigned long long a[4] = {0, 0, 0, 0};
    cudaError_t e = bounds_take_first_bad_here(s, &a[0]);
    if (e == cudaSuccess) e = bounds_take_backward(s, &a[1]);
    if (e == cudaSuccess) e = bounds_take_proj(s, &a[2]);
    if (e == cudaSuccess) e = bounds_take_slots(s, &a[3]);
    if (e != cudaSuccess) return e;
    *addr = 0;
    for (int i = 0; i < 4 && *addr == 0; ++i) *addr = a[i] & ~1ull;  // bit 0 marks "set"
    return cudaSuccess;
}
#endif

}  // namespace sc
