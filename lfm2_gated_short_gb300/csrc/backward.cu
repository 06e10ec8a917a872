// backward.cu -- ShortConv backward for one sequence from a zero state.
//
// Liger-Kernel PR #1317, "Kernel changes / Gated short convolution": the B/C
// gate gradients are fused with the depthwise-conv input gradient in one
// pass, and the weight gradient of all K taps of a channel is reduced
// together (no bias). Here one pass over the rows produces dB, dC and dx and
// accumulates dW in registers:
//   dC_t = dy_t z_t,  dz_t = dy_t C_t,  du_s = sum_k w_k dz_{s+K-1-k},
//   dB_s = du_s x_s,  dx_s = du_s B_s,  dW[h,k] = sum_t dz_t u_{t-K+1+k}.
//
// Thread = (8 channels, a segment of RB consecutive rows). It walks rows
// r0-K+1 .. r1+K-2: the K-1 rows before its segment rebuild the u history,
// the K-1 rows after it supply the dz look-ahead that du needs. The dW
// partial sums of the 8 segments of a CTA are added in shared memory, each
// CTA row writes one [H, K] fp32 partial to the workspace, and a second
// kernel adds the partials in a fixed order (deterministic bits).
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.h"
#include "shortconv.h"

namespace sc {

constexpr int kBwdGroups = 32;   // channel groups per CTA (threadIdx.x): 256 channels
constexpr int kBwdSegs = 8;      // row segments per CTA (threadIdx.y)
constexpr int kBwdChunk = 2;     // rows whose loads are issued together
constexpr int64_t kBwdTargetCtas = 1216;

static int bwd_rows_per_thread(int H, int64_t T) {
    const int64_t gx = (H / kCh + kBwdGroups - 1) / kBwdGroups;
    int64_t rb = (T * gx + kBwdSegs * kBwdTargetCtas - 1) / (kBwdSegs * kBwdTargetCtas);
    if (rb < 4) rb = 4;
    if (rb > 1024) rb = 1024;
    return (int)((rb + 3) / 4 * 4);
}

static int64_t bwd_row_ctas(int H, int64_t T) {
    const int64_t rows_per_cta = (int64_t)kBwdSegs * bwd_rows_per_thread(H, T);
    return (T + rows_per_cta - 1) / rows_per_cta;
}

size_t backward_workspace_bytes(int H, int K, int64_t T) {
    return (size_t)bwd_row_ctas(H, T) * (size_t)H * (size_t)K * sizeof(float);
}

template <typename T, int K>
__global__ void __launch_bounds__(kBwdGroups *kBwdSegs)
    k_backward(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
               const T *__restrict__ dy, T *__restrict__ dbcx, float *__restrict__ partial,
               int RB) {
    constexpr int KH = K > 1 ? K - 1 : 1;  // history / look-ahead depth
    pdl_wait();
    const int groups = H / kCh;
    const int cg = blockIdx.x * kBwdGroups + threadIdx.x;
    const int h0 = cg * kCh;
    const int64_t r0 = ((int64_t)blockIdx.y * kBwdSegs + threadIdx.y) * RB;
    const int64_t r1 = min(r0 + (int64_t)RB, T_rows);
    const int64_t ld = 3 * (int64_t)H;

    float acc[kCh][K];
#pragma unroll
    for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
        for (int k = 0; k < K; ++k) acc[ch][k] = 0.f;

    if (cg < groups && r0 < T_rows) {
        float wt[kCh][K];
        load_block<T, K>(w + (int64_t)h0 * K, wt);
        float uh[kCh][KH], dzq[kCh][KH];  // u and dz of rows t-K+1 .. t-1 (oldest first)
        Row<T> rbq[KH], rxq[KH];         // B and x of rows t-K+1 .. t-1
#pragma unroll
        for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
            for (int k = 0; k < KH; ++k) uh[ch][k] = dzq[ch][k] = 0.f;

        // Rows before the segment: only their u (zero before row 0).
#pragma unroll
        for (int j = 1; j < K; ++j) {
            const int64_t t = r0 - K + j;
            if (t >= 0) {
                const T *p = bcx + t * ld + h0;
                const Row<T> rb = load_row(p), rx = load_row(p + 2 * H);
                float b[kCh], x[kCh];
                unpack_row(rb, b);
                unpack_row(rx, x);
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) uh[ch][j - 1] = gate_in<T>(b[ch], x[ch]);
            }
        }

        // du_s for s = t-K+1 from dz_t and the queued dz, then dB_s, dx_s.
        auto emit = [&](int64_t t, const float (&dz)[kCh], const Row<T> &rb_s,
                        const Row<T> &rx_s) {
            const int64_t s = t - (K - 1);
            if (s < r0) return;
            float b[kCh], x[kCh], db[kCh], dx[kCh];
            unpack_row(rb_s, b);
            unpack_row(rx_s, x);
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch) {
                float du = wt[ch][0] * dz[ch];
#pragma unroll
                for (int k = 1; k < K; ++k) du = fmaf(wt[ch][k], dzq[ch][K - 1 - k], du);
                db[ch] = du * x[ch];
                dx[ch] = du * b[ch];
            }
            T *q = dbcx + s * ld + h0;
            store_row(q, db);
            store_row(q + 2 * H, dx);
        };
        auto push = [&](const float (&u)[kCh], const float (&dz)[kCh], const Row<T> &rb,
                        const Row<T> &rx) {
            if constexpr (K > 1) {
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) {
#pragma unroll
                    for (int k = 0; k + 1 < KH; ++k) {
                        uh[ch][k] = uh[ch][k + 1];
                        dzq[ch][k] = dzq[ch][k + 1];
                    }
                    uh[ch][KH - 1] = u[ch];
                    dzq[ch][KH - 1] = dz[ch];
                }
#pragma unroll
                for (int k = 0; k + 1 < KH; ++k) {
                    rbq[k] = rbq[k + 1];
                    rxq[k] = rxq[k + 1];
                }
                rbq[KH - 1] = rb;
                rxq[KH - 1] = rx;
            }
        };

        // The segment's own rows.
        for (int64_t t0 = r0; t0 < r1; t0 += kBwdChunk) {
            Row<T> lb[kBwdChunk], lc[kBwdChunk], lx[kBwdChunk], lg[kBwdChunk];
#pragma unroll
            for (int j = 0; j < kBwdChunk; ++j) {
                if (t0 + j < r1) {
                    const T *p = bcx + (t0 + j) * ld + h0;
                    lb[j] = load_row(p);
                    lc[j] = load_row(p + H);
                    lx[j] = load_row(p + 2 * H);
                    lg[j] = load_row(dy + (t0 + j) * (int64_t)H + h0);
                }
            }
#pragma unroll
            for (int j = 0; j < kBwdChunk; ++j) {
                const int64_t t = t0 + j;
                if (t < r1) {
                    float b[kCh], c[kCh], x[kCh], g[kCh], u[kCh], dz[kCh], dc[kCh];
                    unpack_row(lb[j], b);
                    unpack_row(lc[j], c);
                    unpack_row(lx[j], x);
                    unpack_row(lg[j], g);
#pragma unroll
                    for (int ch = 0; ch < kCh; ++ch) {
                        u[ch] = gate_in<T>(b[ch], x[ch]);
                        float z = wt[ch][K - 1] * u[ch];
#pragma unroll
                        for (int k = 0; k + 1 < K; ++k) z = fmaf(wt[ch][k], uh[ch][k], z);
                        dc[ch] = g[ch] * z;
                        dz[ch] = g[ch] * c[ch];
#pragma unroll
                        for (int k = 0; k + 1 < K; ++k) acc[ch][k] = fmaf(dz[ch], uh[ch][k], acc[ch][k]);
                        acc[ch][K - 1] = fmaf(dz[ch], u[ch], acc[ch][K - 1]);
                    }
                    store_row(dbcx + t * ld + H + h0, dc);
                    if constexpr (K == 1)
                        emit(t, dz, lb[j], lx[j]);
                    else
                        emit(t, dz, rbq[0], rxq[0]);
                    push(u, dz, lb[j], lx[j]);
                }
            }
        }

        // Rows after the segment: only their dz (zero past the last row).
#pragma unroll
        for (int j = 0; j + 1 < K; ++j) {
            const int64_t t = r1 + j;
            float dz[kCh], u[kCh];
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch) dz[ch] = u[ch] = 0.f;
            if (t < T_rows) {
                const Row<T> rc = load_row(bcx + t * ld + H + h0);
                const Row<T> rg = load_row(dy + t * (int64_t)H + h0);
                float c[kCh], g[kCh];
                unpack_row(rc, c);
                unpack_row(rg, g);
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) dz[ch] = g[ch] * c[ch];
            }
            emit(t, dz, rbq[0], rxq[0]);
            push(u, dz, rbq[0], rxq[0]);
        }
    }

    pdl_launch_dependents();
    // dW: add the 8 segments of this CTA in a fixed order, one partial per CTA row.
    __shared__ float red[kBwdSegs][kBwdGroups * kCh * K];
#pragma unroll
    for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
        for (int k = 0; k < K; ++k) red[threadIdx.y][threadIdx.x * kCh * K + ch * K + k] = acc[ch][k];
    __syncthreads();
    const int tid = threadIdx.y * kBwdGroups + threadIdx.x;
    for (int e = tid; e < kBwdGroups * kCh * K; e += kBwdGroups * kBwdSegs) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < kBwdSegs; ++j) s += red[j][e];
        const int cg2 = blockIdx.x * kBwdGroups + e / (kCh * K);
        if (cg2 < groups)
            partial[(int64_t)blockIdx.y * H * K + (int64_t)cg2 * kCh * K + e % (kCh * K)] = s;
    }
}

// dw[e] = sum over CTA rows g = 0 .. G-1 of partial[g][e], in that order.
__global__ void __launch_bounds__(256)
    k_dw_reduce(const float *__restrict__ partial, int64_t G, int HK, float *__restrict__ dw) {
    pdl_wait();
    pdl_launch_dependents();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= HK) return;
    float s = 0.f;
    for (int64_t g = 0; g < G; ++g) s += partial[g * HK + e];
    dw[e] = s;
}

template <typename T, int K>
static cudaError_t backward_inst(const void *bcx, int64_t rows, int H, const void *w,
                                 const void *dy, void *dbcx, float *dw, void *ws,
                                 cudaStream_t stream) {
    const int RB = bwd_rows_per_thread(H, rows);
    const int64_t gy = bwd_row_ctas(H, rows);
    const int gx = (H / kCh + kBwdGroups - 1) / kBwdGroups;
    if (gy > 0) {
        const cudaError_t e = launch_pdl(
            k_backward<T, K>, dim3(gx, (unsigned)gy), dim3(kBwdGroups, kBwdSegs), 0, stream,
            (const T *)bcx, rows, H, (const T *)w, (const T *)dy, (T *)dbcx, (float *)ws, RB);
        if (e != cudaSuccess) return e;
    }
    const int HK = H * K;
    return launch_pdl(k_dw_reduce, dim3((HK + 255) / 256), dim3(256), 0, stream,
                      (const float *)ws, gy, HK, dw);
}

template <typename T>
static cudaError_t backward_K(int K, const void *bcx, int64_t rows, int H, const void *w,
                              const void *dy, void *dbcx, float *dw, void *ws, cudaStream_t s) {
    switch (K) {
        case 1: return backward_inst<T, 1>(bcx, rows, H, w, dy, dbcx, dw, ws, s);
        case 2: return backward_inst<T, 2>(bcx, rows, H, w, dy, dbcx, dw, ws, s);
        case 3: return backward_inst<T, 3>(bcx, rows, H, w, dy, dbcx, dw, ws, s);
        default: return backward_inst<T, 4>(bcx, rows, H, w, dy, dbcx, dw, ws, s);
    }
}

cudaError_t launch_backward(int dtype, int H, int K, const void *bcx, int64_t rows, const void *w,
                            const void *dy, void *dbcx, float *dw, void *ws, cudaStream_t s) {
    if (dtype == SC_BF16) return backward_K<__nv_bfloat16>(K, bcx, rows, H, w, dy, dbcx, dw, ws, s);
    return backward_K<float>(K, bcx, rows, H, w, dy, dbcx, dw, ws, s);
}

// ------------------------------------------------ no-allocation entry point
//
// shortconv_backward_noalloc runs the kernels above with their fp32 dW
// partials in this fixed device array instead of a caller workspace. It is
// for callers that cannot allocate device memory at call time. It holds
// kNoAllocScratchBytes on every GPU that loads the library, until exit.
// Every entry the reduction reads is first written by the same call, so the
// array needs no clearing; concurrent calls on the same GPU share it and race.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// The array's device address on the current device. In host code the array's
// name is only a host-side stand-in, so the address comes from the runtime:
// once per device (with that device current), then from the cache.
static cudaError_t noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_backward_noalloc(int dtype, int H, int K, const void *bcx, int64_t T,
                                    const void *w, const void *dy, void *dbcx, float *dw,
                                    cudaStream_t s) {
    void *ws = nullptr;
    const cudaError_t e = noalloc_scratch(&ws);
    if (e != cudaSuccess) return e;
    if (dtype == SC_BF16) return backward_K<__nv_bfloat16>(K, bcx, T, H, w, dy, dbcx, dw, ws, s);
    return backward_K<float>(K, bcx, T, H, w, dy, dbcx, dw, ws, s);
}

}  // namespace sc
