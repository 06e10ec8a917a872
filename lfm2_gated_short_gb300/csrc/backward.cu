// backward.cu -- ShortConv backward for one sequence from a zero state.
//
// Liger-Kernel PR #1317, "Kernel changes / Gated short convolution": the B/C
// gate gradients are fused with the depthwise-conv input gradient in one
// pass, and the weight gradient of all K taps of a channel is reduced
// together. One pass over the rows produces dB, dC and dx and accumulates dW
// (and, with the optional conv bias b, dbias) in registers:
//   z_t = sum_k w_k u_{t-K+1+k} (+ b),  dC_t = dy_t z_t,  dz_t = dy_t C_t,
//   du_s = sum_k w_k dz_{s+K-1-k},  dB_s = du_s x_s,  dx_s = du_s B_s,
//   dW[h,k] = sum_t dz_t u_{t-K+1+k},  dbias[h] = sum_t dz_t.
//
// Same streamed design as the prefill: persistent CTAs (several per SM) each
// own a balanced range of rows [cr0, cr1) of a slice of up to 512 channels; a
// producer warp streams the rows' B|C|x and dy sections -- plus the K-1 rows
// before the range (u history) and after it (dz look-ahead) -- through a
// shared-memory ring with 1-D bulk asynchronous copies on full/empty
// mbarriers; the consumer warps, 4 channels per thread, walk the rows. Each
// thread holds its channels' dW (and dbias) over the whole range in registers
// and writes one fp32 partial per CTA; a second kernel adds the partials of
// all CTAs in a fixed order, so dW and dbias have the same bits on every call
// with the same T, H and device (the row split depends on those alone).
// Partial layout per row range: H*K dW entries, then H dbias entries when the
// caller asked for dbias.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "errors.cuh"
#include "kernels.h"
#include "launch.h"
#include "shortconv.h"
#include "tma.cuh"

namespace sc {

// Build-time shape (defaults are the tuned ones): channels per CTA slice and
// the CTAs per SM the register budget is sized for.
#ifndef SC_BWD_SLICE
#define SC_BWD_SLICE 512
#endif
#ifndef SC_BWD_MIN_CTAS
#define SC_BWD_MIN_CTAS 4
#endif
#ifndef SC_BWD_VARLEN_MIN_CTAS
#define SC_BWD_VARLEN_MIN_CTAS 3  // the varlen kernel holds more state per thread
#endif

constexpr int kBwdCpt = 4;                         // channels per consumer thread
constexpr int kBwdSlice = SC_BWD_SLICE;            // channels per CTA slice
constexpr int kBwdConsumers = kBwdSlice / kBwdCpt;
#ifndef SC_BWD_HALO_HINT
#define SC_BWD_HALO_HINT 1  // 1: evict-last L2 policy on the rows a neighbouring CTA reads again
#endif
// Row ranges up to this many rows take the hint. There the K-1 rows before
// and after a range are a sizeable share of its reads (4 of 31 rows at
// T = 4096, H = 2048), and without the hint the second read of them missed
// L2 (T = 4096: 70.6-73.4 MB read per launch for 67.1 MB of inputs; with
// it 65.0-67.2 MB). Longer ranges (T = 65536: 431 rows) do without it: in
// k_backward they run an instance without the hint's code, which measured
// 1% faster there than the same code with the hint switched off at run time.
constexpr int64_t kBwdHintRows = 256;
#ifndef SC_BWD_STAGES
#define SC_BWD_STAGES 4  // stage ring depth (the header holds up to 16 stages' barriers)
#endif
constexpr int kBwdStages = SC_BWD_STAGES;
constexpr int kBwdMinRows = 16;                    // rows per CTA at least
constexpr int kBwdRowCtas = 152;                   // row ranges per slice (GB300: one per SM)
constexpr int kBwdHeader = 256;                    // mbarriers

template <typename T>
struct BwdShape {
    static constexpr int R = sizeof(T) == 2 ? 2 : 1;  // rows per stage (16 / 32 KB per row)
};

template <typename T>
constexpr size_t bwd_smem_bytes(int CW) {
    return (size_t)kBwdHeader + (size_t)kBwdStages * BwdShape<T>::R * 4 * CW * sizeof(T);
}

// CTAs per SM each kernel's registers are budgeted for. K = 4 keeps a fourth
// window tap per channel pair and spilled at the K <= 3 budgets (backward
// 550 us against 313 us at T = 65536), so it is budgeted one CTA fewer.
// fp32 holds twice the bytes per section and takes one CTA fewer again at K = 4.
template <typename T, int K>
constexpr int kBwdCtas = K == 4 ? SC_BWD_MIN_CTAS - (sizeof(T) == 4 ? 2 : 1) : SC_BWD_MIN_CTAS;
template <int K>
constexpr int kBwdVarlenCtas = K == 4 ? SC_BWD_VARLEN_MIN_CTAS - 1 : SC_BWD_VARLEN_MIN_CTAS;

// Row ranges per channel slice at most; fixed by T alone so the workspace
// size is. A launch may use fewer (bwd_launch_rows).
static int64_t bwd_row_ctas(int64_t T) {
    const int64_t n = (T + kBwdMinRows - 1) / kBwdMinRows;
    return n < 1 ? 1 : (n > kBwdRowCtas ? kBwdRowCtas : n);
}

size_t backward_partial_bytes(int H, int K, int64_t T, bool with_dbias) {
    return (size_t)bwd_row_ctas(T) * (size_t)H * (size_t)(K + (with_dbias ? 1 : 0)) *
           sizeof(float);
}

size_t backward_workspace_bytes(int H, int K, int64_t T) {
    return backward_partial_bytes(H, K, T, true);
}

// The conv bias of a thread's CPT channels as pairs (zeros without a bias).
template <typename T, int CPT>
__device__ __forceinline__ void load_bias_pairs(const T *__restrict__ bias, int h0,
                                                f32x2 (&bp)[CPT / 2]) {
#pragma unroll
    for (int q = 0; q < CPT / 2; ++q)
        bp[q] = bias != nullptr
                    ? f2_make(ld_elem(bias + h0 + 2 * q), ld_elem(bias + h0 + 2 * q + 1))
                    : 0ull;
}

// One row range's dW (and dbias) partial for a thread's CPT channels.
template <int K, int CPT>
__device__ __forceinline__ void store_partial(float *__restrict__ part, int H, int h0,
                                              bool with_dbias, const f32x2 (&acc)[K][CPT / 2],
                                              const f32x2 (&accb)[CPT / 2]) {
    float *pp = part + (int64_t)h0 * K;
#pragma unroll
    for (int q = 0; q < CPT / 2; ++q) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float lo, hi;
            f2_split(acc[k][q], lo, hi);
            gst(pp + (2 * q) * K + k, lo);
            gst(pp + (2 * q + 1) * K + k, hi);
        }
        if (with_dbias) {
            float lo, hi;
            f2_split(accb[q], lo, hi);
            gst(part + (int64_t)H * K + h0 + 2 * q, lo);
            gst(part + (int64_t)H * K + h0 + 2 * q + 1, hi);
        }
    }
}

// HB: a conv bias is given or dbias is wanted. The instance without carries
// no bias registers or branches; with_dbias then is false.
template <typename T, int K, bool HB, bool HINT>
__global__ void __launch_bounds__(kBwdConsumers + 32, kBwdCtas<T, K>)
    k_backward(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
               const T *__restrict__ bias, const T *__restrict__ dy, T *__restrict__ dbcx,
               float *__restrict__ partial, bool with_dbias, int n_slices, int n_row_ctas) {
    constexpr int CPT = kBwdCpt;
    constexpr int NP = CPT / 2;
    constexpr int R = BwdShape<T>::R;
    constexpr int NS = kBwdStages;
    constexpr int KH = K > 1 ? K - 1 : 1;  // history / look-ahead depth
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + 128);
    T *stage = reinterpret_cast<T *>(smem + kBwdHeader);

    const int tid = threadIdx.x;
    const int n_consumers = blockDim.x - 32;
    const bool producer = tid >= n_consumers;
    const bool lead = tid == n_consumers;
    const int slice = blockIdx.x % n_slices;
    const int64_t rc = blockIdx.x / n_slices;
    const int c0 = slice * kBwdSlice;
    const int CW = min(kBwdSlice, H);
    const int cw = min(kBwdSlice, H - c0);
    const bool active = !producer && tid * CPT < cw;
    const int h0 = c0 + tid * CPT;
    const int64_t cr0 = rc * T_rows / n_row_ctas, cr1 = (rc + 1) * T_rows / n_row_ctas;
    const int64_t sr0 = max((int64_t)0, cr0 - (K - 1));
    const int64_t sr1 = min(T_rows, cr1 + (K - 1));
    const int n_chunks = cr0 < cr1 ? (int)((sr1 - sr0 + R - 1) / R) : 0;
    const uint32_t sec_bytes = (uint32_t)cw * sizeof(T);
    const int64_t ld = 3 * (int64_t)H;

    if (lead) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumers / 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();  // inputs may come from the previous kernel in the stream
    pdl_launch_dependents();

    // Stage layout per row: B | C | x | dy sections of CW channels.
    // The 2 (K-1) rows around the range's start are read again by the CTA of
    // the range before, at its end: in the HINT instance (short ranges) they
    // are fetched with an evict-last L2 policy so that second read finds
    // them in L2. Long ranges run the instance without the hint's code.
    const bool hint = HINT && rc > 0;
    const uint64_t keep = hint ? l2_policy_evict_last() : 0;
    auto issue = [&](int c) {
        const int s = c % NS;
        const int64_t rb = sr0 + (int64_t)c * R;
        const int rows = (int)min((int64_t)R, sr1 - rb);
        mbar_arrive_expect_tx(&full[s], (uint32_t)rows * 4u * sec_bytes);
        for (int rr = 0; rr < rows; ++rr) {
            const T *src = bcx + (rb + rr) * ld + c0;
            T *dst = stage + (size_t)(s * R + rr) * 4 * CW;
            if (hint && rb + rr < cr0 + (K - 1)) {
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    bulk_copy_g2s_hint(dst + (size_t)q * CW, src + (int64_t)q * H, sec_bytes,
                                       &full[s], keep);
                bulk_copy_g2s_hint(dst + (size_t)3 * CW, dy + (rb + rr) * (int64_t)H + c0,
                                   sec_bytes, &full[s], keep);
                continue;
            }
#pragma unroll
            for (int q = 0; q < 3; ++q)
                bulk_copy_g2s(dst + (size_t)q * CW, src + (int64_t)q * H, sec_bytes, &full[s]);
            bulk_copy_g2s(dst + (size_t)3 * CW, dy + (rb + rr) * (int64_t)H + c0, sec_bytes,
                          &full[s]);
        }
    };
    auto drain = [&](int from, int to) {
        for (int c = from; c < to; ++c) mbar_wait_bounded(&full[c % NS], (uint32_t)(c / NS) & 1u);
    };

    if (producer) {
        if (!lead) return;
        int c = 0;
        for (; c < n_chunks; ++c) {
            if (c >= NS && !mbar_wait_bounded(&empty[c % NS], (uint32_t)(c / NS - 1) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                break;
            }
            issue(c);
        }
        drain(max(0, c - NS), c);
        return;
    }

    f32x2 wp[K][NP], bp[NP], accb[NP];  // taps, conv bias, dbias
    if (active) {
        load_taps<T, CPT, K>(w + (int64_t)h0 * K, wp);
        if constexpr (HB) load_bias_pairs<T, CPT>(bias, h0, bp);
    }
    f32x2 uw[K][NP], dzw[K][NP], acc[K][NP];  // u window, dz window (newest last), dW
    Sec<T, CPT> rbq[KH], rxq[KH];             // B and x of the K-1 rows before t
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        accb[q] = 0ull;
#pragma unroll
        for (int k = 0; k < K; ++k) uw[k][q] = dzw[k][q] = acc[k][q] = 0ull;
    }
    const f32x2 one2 = f2_make(1.f, 1.f);

    // du for row s = t-K+1 from the dz window (dz_t newest), then dB_s, dx_s.
    auto emit = [&](int64_t t, const Sec<T, CPT> &b_s, const Sec<T, CPT> &x_s) {
        const int64_t s = t - (K - 1);
        if (s < cr0 || s >= cr1) return;
        f32x2 fb[NP], fx[NP], db[NP], dx[NP];
        Pairs<T, CPT>::widen(b_s, fb);
        Pairs<T, CPT>::widen(x_s, fx);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            f32x2 du = f2_mul(wp[0][q], dzw[K - 1][q]);
#pragma unroll
            for (int k = 1; k < K; ++k) du = f2_fma(wp[k][q], dzw[K - 1 - k][q], du);
            db[q] = f2_mul(du, fx[q]);
            dx[q] = f2_mul(du, fb[q]);
        }
        T *o = dbcx + s * ld + h0;
        Pairs<T, CPT>::store(o, db);
        Pairs<T, CPT>::store(o + 2 * H, dx);
    };
    auto push_bx = [&](const Sec<T, CPT> &b, const Sec<T, CPT> &x) {
        if constexpr (K > 1) {
#pragma unroll
            for (int k = 0; k + 1 < KH; ++k) {
                rbq[k] = rbq[k + 1];
                rxq[k] = rxq[k + 1];
            }
            rbq[KH - 1] = b;
            rxq[KH - 1] = x;
        }
    };
    auto slide = [&](f32x2 (&win)[K][NP], const f32x2 (&v)[NP]) {
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int k = 0; k + 1 < K; ++k) win[k][q] = win[k + 1][q];
            win[K - 1][q] = v[q];
        }
    };

    const int lane = tid & 31;
    const uint32_t base = smem_addr(stage) + (uint32_t)(tid * CPT * sizeof(T));
    const uint32_t sec = (uint32_t)(CW * sizeof(T));
    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % NS;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(c / NS) & 1u)) {
            if (lane == 0) raise_error(SC_DEV_TIMEOUT);
            return;
        }
        const int64_t rb = sr0 + (int64_t)c * R;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int64_t t = rb + rr;
            if (t >= sr1) break;
            if (!active) continue;
            const uint32_t a = base + (uint32_t)((s * R + rr) * 4) * sec;
            const Sec<T, CPT> b = lds_sec<T, CPT>(a), x = lds_sec<T, CPT>(a + 2 * sec);
            const Sec<T, CPT> cc = lds_sec<T, CPT>(a + sec), g = lds_sec<T, CPT>(a + 3 * sec);
            f32x2 u[NP], fc[NP], fg[NP], dz[NP];
            Pairs<T, CPT>::gate(b, x, u);
            Pairs<T, CPT>::widen(cc, fc);
            Pairs<T, CPT>::widen(g, fg);
#pragma unroll
            for (int q = 0; q < NP; ++q) dz[q] = f2_mul(fg[q], fc[q]);
            slide(uw, u);
            slide(dzw, dz);
            if (t >= cr0 && t < cr1) {
                f32x2 dc[NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    f32x2 z = f2_mul(wp[0][q], uw[0][q]);  // the forward's order
#pragma unroll
                    for (int k = 1; k < K; ++k) z = f2_fma(wp[k][q], uw[k][q], z);
                    if constexpr (HB)
                        if (bias != nullptr) z = f2_fma(one2, bp[q], z);
                    dc[q] = f2_mul(fg[q], z);
#pragma unroll
                    for (int k = 0; k < K; ++k) acc[k][q] = f2_fma(dz[q], uw[k][q], acc[k][q]);
                    if constexpr (HB) accb[q] = f2_fma(one2, dz[q], accb[q]);
                }
                Pairs<T, CPT>::store(dbcx + t * ld + H + h0, dc);
            }
            if constexpr (K == 1)
                emit(t, b, x);
            else
                emit(t, rbq[0], rxq[0]);
            push_bx(b, x);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!active) return;
    // Rows past the last one have dz = 0: finish the last K-1 emissions.
#pragma unroll
    for (int j = 0; j + 1 < K; ++j) {
        const int64_t t = sr1 + j;
        if (cr0 >= cr1 || t >= cr1 + (K - 1)) break;
        f32x2 zero[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) zero[q] = 0ull;
        slide(dzw, zero);
        emit(t, rbq[0], rxq[0]);
        push_bx(rbq[0], rxq[0]);
    }
    // This CTA's dW (and dbias) partial for its channels (zero for an empty range).
    store_partial<K, CPT>(partial + rc * (int64_t)H * (K + (with_dbias ? 1 : 0)), H, h0,
                          HB && with_dbias, acc, accb);
}

// ------------------------------------------------ packed varlen, with states
//
// The backward of the packed varlen prefill (rows cu[i] .. cu[i+1]-1 form
// sequence i) with initial states init[i] and an optional gradient d_final[i]
// flowing in through each sequence's final state. Per sequence, with
// ext = [init_0 .. init_{K-1}, u_0 .. u_{len-1}], row t's window is
// ext[t+1 .. t+K]; du_s sums w_k dz over rows of the same sequence only, plus
// d_final[K + s - s1] for the last K rows; d_init[i][m] = sum_{k<m} w_k dz_{m-1-k}
// (+ d_final[m - len] when m >= len).
// Work split as in k_backward. A thread follows the sequence pieces of its
// CTA's stream: a sequence starting inside the stream takes its window from
// its initial state; at a sequence end K-1 virtual rows with dz = 0 finish the
// last emissions; the CTA holding a sequence's first row (its owner) writes
// d_init from the dz of the sequence's first K-1 rows, recorded on the way.
// Empty sequences get d_init = d_final from the CTA whose range holds their
// start (the last CTA for those starting at T).
constexpr int kBwdStaged = 512;  // cu_seqlens entries staged in shared memory
constexpr int kBwdCuBytes = ((kBwdStaged + 1) * 4 + 127) / 128 * 128;

template <typename T>
constexpr size_t bwd_varlen_smem_bytes(int CW) {
    return bwd_smem_bytes<T>(CW) + kBwdCuBytes;
}

template <typename T, int K, bool HB>
__global__ void __launch_bounds__(kBwdConsumers + 32, kBwdVarlenCtas<K>)
    k_backward_varlen(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
                      const T *__restrict__ bias, const int32_t *__restrict__ cu, int N,
                      const T *__restrict__ init, const T *__restrict__ dy,
                      const float *__restrict__ d_final, T *__restrict__ dbcx,
                      float *__restrict__ partial, bool with_dbias, float *__restrict__ d_init,
                      int n_slices, int n_row_ctas) {
    constexpr int CPT = kBwdCpt;
    constexpr int NP = CPT / 2;
    constexpr int R = BwdShape<T>::R;
    constexpr int NS = kBwdStages;
    constexpr int KH = K > 1 ? K - 1 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + 128);
    int32_t *s_cu = reinterpret_cast<int32_t *>(smem + kBwdHeader);
    T *stage = reinterpret_cast<T *>(smem + kBwdHeader + kBwdCuBytes);

    const int tid = threadIdx.x;
    const int n_consumers = blockDim.x - 32;
    const bool producer = tid >= n_consumers;
    const bool lead = tid == n_consumers;
    const int slice = blockIdx.x % n_slices;
    const int64_t rc = blockIdx.x / n_slices;
    const int c0 = slice * kBwdSlice;
    const int CW = min(kBwdSlice, H);
    const int cw = min(kBwdSlice, H - c0);
    const bool active = !producer && tid * CPT < cw;
    const int h0 = c0 + tid * CPT;
    const int64_t cr0 = rc * T_rows / n_row_ctas, cr1 = (rc + 1) * T_rows / n_row_ctas;
    const int64_t sr0 = max((int64_t)0, cr0 - (K - 1));
    const int64_t sr1 = min(T_rows, cr1 + (K - 1));
    const int n_chunks = cr0 < cr1 ? (int)((sr1 - sr0 + R - 1) / R) : 0;
    const uint32_t sec_bytes = (uint32_t)cw * sizeof(T);
    const int64_t ld = 3 * (int64_t)H;
    float *part = partial + rc * (int64_t)H * (K + (with_dbias ? 1 : 0));

    if (lead) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumers / 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    // Evict-last L2 policy on the rows around the range's start, which the
    // CTA before reads again at its end (as in k_backward).
    const bool hint = SC_BWD_HALO_HINT && rc > 0 && cr1 - cr0 <= kBwdHintRows;
    const uint64_t keep = hint ? l2_policy_evict_last() : 0;
    auto issue = [&](int c) {
        const int s = c % NS;
        const int64_t rb = sr0 + (int64_t)c * R;
        const int rows = (int)min((int64_t)R, sr1 - rb);
        mbar_arrive_expect_tx(&full[s], (uint32_t)rows * 4u * sec_bytes);
        for (int rr = 0; rr < rows; ++rr) {
            const T *src = bcx + (rb + rr) * ld + c0;
            T *dst = stage + (size_t)(s * R + rr) * 4 * CW;
            if (hint && rb + rr < cr0 + (K - 1)) {
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    bulk_copy_g2s_hint(dst + (size_t)q * CW, src + (int64_t)q * H, sec_bytes,
                                       &full[s], keep);
                bulk_copy_g2s_hint(dst + (size_t)3 * CW, dy + (rb + rr) * (int64_t)H + c0,
                                   sec_bytes, &full[s], keep);
                continue;
            }
#pragma unroll
            for (int q = 0; q < 3; ++q)
                bulk_copy_g2s(dst + (size_t)q * CW, src + (int64_t)q * H, sec_bytes, &full[s]);
            bulk_copy_g2s(dst + (size_t)3 * CW, dy + (rb + rr) * (int64_t)H + c0, sec_bytes,
                          &full[s]);
        }
    };
    auto drain = [&](int from, int to) {
        for (int c = from; c < to; ++c) mbar_wait_bounded(&full[c % NS], (uint32_t)(c / NS) & 1u);
    };
    const int first = min(NS, n_chunks);
    if (lead)
        for (int c = 0; c < first; ++c) issue(c);

    const bool staged = N <= kBwdStaged;
    int bad = 0;
    for (int j = tid; j <= N; j += blockDim.x) {
        const int32_t c = gld(cu + j);
        if (staged) s_cu[j] = c;
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && gld(cu + j + 1) < c) bad = 1;
    }
    f32x2 acc[K][NP], accb[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        accb[q] = 0ull;
#pragma unroll
        for (int k = 0; k < K; ++k) acc[k][q] = 0ull;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && tid == 0) raise_error(SC_DEV_BAD_SEQLENS);
        if (lead) drain(0, first);
        // dW and dbias become 0; dB|dC|dx and d_init are not written
        if (active) store_partial<K, CPT>(part, H, h0, HB && with_dbias, acc, accb);
        return;
    }

    if (producer) {
        if (!lead) return;
        int c = first;
        for (; c < n_chunks; ++c) {
            if (!mbar_wait_bounded(&empty[c % NS], (uint32_t)(c / NS - 1) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                break;
            }
            issue(c);
        }
        drain(max(0, c - NS), c);
        return;
    }

    auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : gld(cu + j); };
    f32x2 wp[K][NP], bp[NP];
    if (active) {
        load_taps<T, CPT, K>(w + (int64_t)h0 * K, wp);
        if constexpr (HB) load_bias_pairs<T, CPT>(bias, h0, bp);
    }
    const f32x2 one2 = f2_make(1.f, 1.f);
    f32x2 uw[K][NP], dzw[K][NP], dfin[K][NP];
    Sec<T, CPT> rbq[KH], rxq[KH];
    int i = 0;
    int64_t s0 = 0, s1 = 0;
    bool owner = false;

    auto zero = [&](auto &a) {
        for (auto &row : a)
#pragma unroll
            for (int q = 0; q < NP; ++q) row[q] = 0ull;
    };
    auto enter = [&]() {
        owner = s0 >= cr0 && s0 < cr1;
        if (s0 >= sr0 && init != nullptr)
            load_taps<T, CPT, K>(init + ((int64_t)i * H + h0) * K, uw);
        else
            zero(uw);
        zero(dzw);
        if (d_final != nullptr && s1 - K < cr1)  // needed only for the last K rows
            load_taps<float, CPT, K>(d_final + ((int64_t)i * H + h0) * K, dfin);
        else
            zero(dfin);
    };
    auto slide = [&](f32x2 (&win)[K][NP], const f32x2 (&v)[NP]) {
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int k = 0; k + 1 < K; ++k) win[k][q] = win[k + 1][q];
            win[K - 1][q] = v[q];
        }
    };
    auto push_bx = [&](const Sec<T, CPT> &b, const Sec<T, CPT> &x) {
        if constexpr (K > 1) {
#pragma unroll
            for (int k = 0; k + 1 < KH; ++k) {
                rbq[k] = rbq[k + 1];
                rxq[k] = rxq[k + 1];
            }
            rbq[KH - 1] = b;
            rxq[KH - 1] = x;
        }
    };
    // du for row s = t-K+1 of the current sequence, then dB_s, dx_s.
    auto emit = [&](int64_t t, const Sec<T, CPT> &b_s, const Sec<T, CPT> &x_s, bool fin) {
        const int64_t s = t - (K - 1);
        if (s < s0 || s < cr0 || s >= cr1) return;
        f32x2 fb[NP], fx[NP], db[NP], dx[NP];
        Pairs<T, CPT>::widen(b_s, fb);
        Pairs<T, CPT>::widen(x_s, fx);
        const int64_t f = K + s - s1;  // final-state tap fed by u_s, if in range
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            f32x2 du = f2_mul(wp[0][q], dzw[K - 1][q]);
#pragma unroll
            for (int k = 1; k < K; ++k) du = f2_fma(wp[k][q], dzw[K - 1 - k][q], du);
            if (fin)  // one of the sequence's last K rows may feed the final state
#pragma unroll
                for (int k = 0; k < K; ++k)
                    if (f == k) du = f2_fma(f2_make(1.f, 1.f), dfin[k][q], du);
            db[q] = f2_mul(du, fx[q]);
            dx[q] = f2_mul(du, fb[q]);
        }
        T *o = dbcx + s * ld + h0;
        Pairs<T, CPT>::store(o, db);
        Pairs<T, CPT>::store(o + 2 * H, dx);
    };
    auto write_d_init = [&]() {
        const int64_t len = s1 - s0;
        // dz of the sequence's first K-1 rows (zero past its end), read back
        // from global memory: dy * C rounded once in fp32, as in the row loop.
        f32x2 dzf[KH][NP];
#pragma unroll
        for (int k = 0; k < KH; ++k)
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                dzf[k][q] = 0ull;
                if (K > 1 && k < len) {
                    const T *cp = bcx + (s0 + k) * ld + H + h0 + 2 * q;
                    const T *gp = dy + (s0 + k) * (int64_t)H + h0 + 2 * q;
                    dzf[k][q] = f2_mul(f2_make(ld_elem(gp), ld_elem(gp + 1)),
                                       f2_make(ld_elem(cp), ld_elem(cp + 1)));
                }
            }
        float *o = d_init + ((int64_t)i * H + h0) * K;
#pragma unroll
        for (int q = 0; q < NP; ++q)
#pragma unroll
            for (int m = 0; m < K; ++m) {
                f32x2 g = 0ull;
#pragma unroll
                for (int k = 0; k < m; ++k) g = f2_fma(wp[k][q], dzf[m - 1 - k][q], g);
#pragma unroll
                for (int e = 0; e < K; ++e)  // final-state tap m - len (no runtime index)
                    if (m >= len && e == m - len)
                        g = f2_fma(f2_make(1.f, 1.f), dfin[e][q], g);
                float lo, hi;
                f2_split(g, lo, hi);
                gst(o + (2 * q) * K + m, lo);
                gst(o + (2 * q + 1) * K + m, hi);
            }
    };
    // The sequence ended at s1 inside the stream: K-1 rows with dz = 0 finish
    // its emissions; its owner writes d_init.
    auto finish = [&]() {
        f32x2 zz[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) zz[q] = 0ull;
#pragma unroll
        for (int j = 0; j + 1 < K; ++j) {
            slide(dzw, zz);
            emit(s1 + j, rbq[0], rxq[0], true);
            push_bx(rbq[0], rxq[0]);
        }
        if (owner && d_init != nullptr) write_d_init();
    };

    if (n_chunks > 0 && active) {
        int lo = 0, hi = N - 1;  // largest i with cu[i] <= sr0: the sequence holding row sr0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (CU(mid) <= sr0) lo = mid; else hi = mid - 1;
        }
        i = lo;
        s0 = CU(i);
        s1 = CU(i + 1);
        enter();
    }

    const int lane = tid & 31;
    const uint32_t base = smem_addr(stage) + (uint32_t)(tid * CPT * sizeof(T));
    const uint32_t sec = (uint32_t)(CW * sizeof(T));
    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % NS;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(c / NS) & 1u)) {
            if (lane == 0) raise_error(SC_DEV_TIMEOUT);
            return;
        }
        const int64_t rb = sr0 + (int64_t)c * R;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int64_t t = rb + rr;
            if (t >= sr1) break;
            if (!active) continue;
            if (t >= s1) {
                finish();
                do {
                    ++i;
                    s0 = CU(i);
                    s1 = CU(i + 1);
                } while (t >= s1);
                enter();
            }
            const uint32_t a = base + (uint32_t)((s * R + rr) * 4) * sec;
            const Sec<T, CPT> b = lds_sec<T, CPT>(a), x = lds_sec<T, CPT>(a + 2 * sec);
            const Sec<T, CPT> cc = lds_sec<T, CPT>(a + sec), g = lds_sec<T, CPT>(a + 3 * sec);
            f32x2 u[NP], fc[NP], fg[NP], dz[NP];
            Pairs<T, CPT>::gate(b, x, u);
            Pairs<T, CPT>::widen(cc, fc);
            Pairs<T, CPT>::widen(g, fg);
#pragma unroll
            for (int q = 0; q < NP; ++q) dz[q] = f2_mul(fg[q], fc[q]);
            slide(uw, u);
            slide(dzw, dz);
            if (t >= cr0 && t < cr1) {
                f32x2 dc[NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    f32x2 z = f2_mul(wp[0][q], uw[0][q]);
#pragma unroll
                    for (int k = 1; k < K; ++k) z = f2_fma(wp[k][q], uw[k][q], z);
                    if constexpr (HB)
                        if (bias != nullptr) z = f2_fma(one2, bp[q], z);
                    dc[q] = f2_mul(fg[q], z);
#pragma unroll
                    for (int k = 0; k < K; ++k) acc[k][q] = f2_fma(dz[q], uw[k][q], acc[k][q]);
                    if constexpr (HB) accb[q] = f2_fma(one2, dz[q], accb[q]);
                }
                Pairs<T, CPT>::store(dbcx + t * ld + H + h0, dc);
            }
            const bool fin = t + 1 == s1;  // the sequence's last row: its tap feeds the state
            if constexpr (K == 1)
                emit(t, b, x, fin);
            else
                emit(t, rbq[0], rxq[0], fin);
            push_bx(b, x);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!active) return;
    if (n_chunks > 0) {
        if (s1 <= sr1)
            finish();
        else if (owner && d_init != nullptr)
            write_d_init();  // its first K-1 rows were streamed; the rest is another CTA's
    }
    // Empty sequences starting in this CTA's range (or at T, for the last CTA).
    if (d_init != nullptr) {
        int lo = 0, hi = N;  // first j with cu[j] >= cr0
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (CU(mid) < cr0) lo = mid + 1; else hi = mid;
        }
        const bool last = rc == n_row_ctas - 1;
        for (int j = lo; j < N && (CU(j) < cr1 || (last && CU(j) == T_rows)); ++j) {
            if (CU(j + 1) != CU(j)) continue;
            float *o = d_init + ((int64_t)j * H + h0) * K;
            for (int e = 0; e < CPT * K; ++e)
                gst(o + e, d_final != nullptr ? gld(d_final + ((int64_t)j * H + h0) * K + e) : 0.f);
        }
    }
    store_partial<K, CPT>(part, H, h0, HB && with_dbias, acc, accb);
}

// out[e] = sum over row ranges g = 0 .. G-1 of partial[g][e] for the P
// entries of a partial (dW's HK first, then dbias's): 8 warps take interleaved
// g for 32 consecutive e, then warp 0 adds the 8 sums in order. A thread's
// (at most kRedPerWarp) partials are all requested before the first add, so
// the call costs one memory round trip, not one per partial.
constexpr int kRedPerWarp = (kBwdRowCtas + 7) / 8;
__global__ void __launch_bounds__(256)
    k_dw_reduce(const float *__restrict__ partial, int64_t G, int HK, int P,
                float *__restrict__ dw, float *__restrict__ dbias) {
    __shared__ float part[8][32];
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    float v[kRedPerWarp];
#pragma unroll
    for (int j = 0; j < kRedPerWarp; ++j) {
        const int64_t g = warp + 8 * j;
        v[j] = e < P && g < G ? gld(partial + g * P + e) : 0.f;
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kRedPerWarp; ++j)
        if (warp + 8 * j < G) s += v[j];
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && e < P) {
        float t = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) t += part[j][lane];
        if (e < HK)
            gst(dw + e, t);
        else
            gst(dbias + (e - HK), t);
    }
}

// Row ranges per slice for one launch: one wave of CTAs at the kernel's
// occupancy on this device (n_slices slices share the SMs), capped by what
// the workspace holds. The row split, and so dW's summation order, depends
// only on T, H and the device.
//
// The caller's cache (one per kernel instance) keeps the last (device, slice
// count, slice width) and its wave in one 64-bit word, so concurrent callers
// never pair a key with another key's wave.
struct WaveCache {
    std::atomic<unsigned long long> packed{0};  // key << 20 | wave; 0 = empty
};
template <typename Kern>
static cudaError_t bwd_launch_rows(Kern kern, int threads, size_t smem, int n_slices, int CW,
                                   int64_t T, WaveCache &cache, int64_t *n_row) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long key = ((unsigned long long)(dev & 0xFF) << 36) |
                                   ((unsigned long long)(n_slices & 0xFFFFFF) << 12) |
                                   (unsigned long long)((CW / 8) & 0xFFF);
    const unsigned long long got = cache.packed.load();
    int wave = got != 0 && (got >> 20) == key ? (int)(got & 0xFFFFF) : 0;
    if (wave <= 0) {
        int sms = 0, occ = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
        if (e != cudaSuccess) return e;
        wave = sms * (occ > 0 ? occ : 1) / n_slices;
        if (wave < 1) wave = 1;
        if (wave > 0xFFFFF) wave = 0xFFFFF;
        cache.packed.store(key << 20 | (unsigned long long)wave);
    }
    const int64_t cap = bwd_row_ctas(T);
    *n_row = wave < cap ? wave : cap;
    return cudaSuccess;
}

static cudaError_t launch_reduce(const void *ws, int64_t n_row, int H, int K, float *dw,
                                 float *dbias, cudaStream_t stream) {
    const int HK = H * K, P = HK + (dbias != nullptr ? H : 0);
    return launch_pdl(k_dw_reduce, dim3((unsigned)((P + 31) / 32)), dim3(256), 0, stream,
                      (const float *)ws, n_row, HK, P, dw, dbias);
}

template <typename T, int K, bool HB>
static cudaError_t backward_inst(const void *bcx, int64_t rows, int H, const void *w,
                                 const void *bias, const void *dy, void *dbcx, float *dw,
                                 float *dbias, void *ws, cudaStream_t stream) {
    const int CW = H < kBwdSlice ? H : kBwdSlice;
    const int n_slices = (H + kBwdSlice - 1) / kBwdSlice;
    const int threads = (CW / kBwdCpt + 31) / 32 * 32 + 32;  // consumers + one producer warp
    const size_t smem = bwd_smem_bytes<T>(CW);
    auto kern = k_backward<T, K, HB, false>;
    auto kern_hint = k_backward<T, K, HB, SC_BWD_HALO_HINT != 0>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(configured.load() & (1ull << dev))) {
        for (auto kr : {kern, kern_hint}) {
            e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)bwd_smem_bytes<T>(kBwdSlice));
            if (e != cudaSuccess) return e;
        }
        configured.fetch_or(1ull << dev);
    }
    static WaveCache waves;
    int64_t n_row = 1;
    e = bwd_launch_rows(kern, threads, smem, n_slices, CW, rows, waves, &n_row);
    if (e != cudaSuccess) return e;
    // Both instances have the same register budget and shared memory, so the
    // same row split (and so the same dW bits).
    const bool short_ranges = (rows + n_row - 1) / n_row <= kBwdHintRows;
    e = launch_pdl(short_ranges ? kern_hint : kern, dim3((unsigned)(n_row * n_slices)), dim3(threads), smem, stream,
                   (const T *)bcx, rows, H, (const T *)w, (const T *)bias, (const T *)dy,
                   (T *)dbcx, (float *)ws, dbias != nullptr, n_slices, (int)n_row);
    if (e != cudaSuccess) return e;
    return launch_reduce(ws, n_row, H, K, dw, dbias, stream);
}

template <typename T, int K, bool HB>
static cudaError_t backward_varlen_inst(const void *bcx, int64_t rows, int H, const void *w,
                                        const void *bias, const int32_t *cu, int N,
                                        const void *init, const void *dy, const float *d_final,
                                        void *dbcx, float *dw, float *dbias, float *d_init,
                                        void *ws, cudaStream_t stream) {
    const int CW = H < kBwdSlice ? H : kBwdSlice;
    const int n_slices = (H + kBwdSlice - 1) / kBwdSlice;
    const int threads = (CW / kBwdCpt + 31) / 32 * 32 + 32;
    const size_t smem = bwd_varlen_smem_bytes<T>(CW);
    auto kern = k_backward_varlen<T, K, HB>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(configured.load() & (1ull << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwd_varlen_smem_bytes<T>(kBwdSlice));
        if (e != cudaSuccess) return e;
        configured.fetch_or(1ull << dev);
    }
    static WaveCache waves;
    int64_t n_row = 1;
    e = bwd_launch_rows(kern, threads, smem, n_slices, CW, rows, waves, &n_row);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3((unsigned)(n_row * n_slices)), dim3(threads), smem, stream,
                   (const T *)bcx, rows, H, (const T *)w, (const T *)bias, cu, N,
                   (const T *)init, (const T *)dy, d_final, (T *)dbcx, (float *)ws,
                   dbias != nullptr, d_init, n_slices, (int)n_row);
    if (e != cudaSuccess) return e;
    return launch_reduce(ws, n_row, H, K, dw, dbias, stream);
}

#define SC_VARLEN_ARGS bcx, rows, H, w, bias, cu, N, init, dy, d_final, dbcx, dw, dbias, d_init, ws, s
template <typename T>
static cudaError_t backward_varlen_K(int K, const void *bcx, int64_t rows, int H, const void *w,
                                     const void *bias, const int32_t *cu, int N,
                                     const void *init, const void *dy, const float *d_final,
                                     void *dbcx, float *dw, float *dbias, float *d_init, void *ws,
                                     cudaStream_t s) {
    const bool hb = bias != nullptr || dbias != nullptr;
#define SC_VARLEN_CASE(k)                                                        \
    return hb ? backward_varlen_inst<T, k, true>(SC_VARLEN_ARGS)                 \
              : backward_varlen_inst<T, k, false>(SC_VARLEN_ARGS)
    switch (K) {
        case 1: SC_VARLEN_CASE(1);
        case 2: SC_VARLEN_CASE(2);
        case 3: SC_VARLEN_CASE(3);
        default: SC_VARLEN_CASE(4);
    }
#undef SC_VARLEN_CASE
}
#undef SC_VARLEN_ARGS

cudaError_t launch_backward_varlen(int dtype, int H, int K, const void *bcx, int64_t T,
                                   const void *w, const void *bias, const int32_t *cu, int N,
                                   const void *init, const void *dy, const float *d_final,
                                   void *dbcx, float *dw, float *dbias, float *d_init, void *ws,
                                   cudaStream_t s) {
    if (dtype == SC_BF16)
        return backward_varlen_K<__nv_bfloat16>(K, bcx, T, H, w, bias, cu, N, init, dy, d_final,
                                                dbcx, dw, dbias, d_init, ws, s);
    return backward_varlen_K<float>(K, bcx, T, H, w, bias, cu, N, init, dy, d_final, dbcx, dw,
                                    dbias, d_init, ws, s);
}

template <typename T>
static cudaError_t backward_K(int K, const void *bcx, int64_t rows, int H, const void *w,
                              const void *bias, const void *dy, void *dbcx, float *dw,
                              float *dbias, void *ws, cudaStream_t s) {
    const bool hb = bias != nullptr || dbias != nullptr;
#define SC_BWD_ARGS bcx, rows, H, w, bias, dy, dbcx, dw, dbias, ws, s
#define SC_BWD_CASE(k)                                                         \
    return hb ? backward_inst<T, k, true>(SC_BWD_ARGS) : backward_inst<T, k, false>(SC_BWD_ARGS)
    switch (K) {
        case 1: SC_BWD_CASE(1);
        case 2: SC_BWD_CASE(2);
        case 3: SC_BWD_CASE(3);
        default: SC_BWD_CASE(4);
    }
#undef SC_BWD_CASE
#undef SC_BWD_ARGS
}

cudaError_t launch_backward(int dtype, int H, int K, const void *bcx, int64_t T, const void *w,
                            const void *bias, const void *dy, void *dbcx, float *dw,
                            float *dbias, void *ws, cudaStream_t s) {
    if (dtype == SC_BF16)
        return backward_K<__nv_bfloat16>(K, bcx, T, H, w, bias, dy, dbcx, dw, dbias, ws, s);
    return backward_K<float>(K, bcx, T, H, w, bias, dy, dbcx, dw, dbias, ws, s);
}

cudaError_t take_error_backward(cudaStream_t stream, unsigned int *code) {
    return take_error_here(stream, code);
}

#ifdef SC_BOUNDS_CHECK
cudaError_t bounds_install_backward(const BoundsRegion *r, int n, cudaStream_t stream) {
    return bounds_install_here(r, n, stream);
}
cudaError_t bounds_take_backward(cudaStream_t stream, unsigned long long *addr) {
    return bounds_take_first_bad_here(stream, addr);
}
#endif

// ------------------------------------------------ no-allocation entry point
//
// shortconv_backward_noalloc runs the kernels above (without a conv bias) with
// their fp32 dW partials in this fixed device array instead of a caller
// workspace. It is
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
    cudaError_t e = noalloc_scratch(&ws);
    if (e != cudaSuccess) return e;
#ifdef SC_BOUNDS_CHECK
    e = bounds_append_here(BoundsRegion{reinterpret_cast<uint64_t>(ws), kNoAllocScratchBytes, 1, 0},
                           s);
    if (e != cudaSuccess) return e;
#endif
    if (dtype == SC_BF16)
        return backward_K<__nv_bfloat16>(K, bcx, T, H, w, nullptr, dy, dbcx, dw, nullptr, ws, s);
    return backward_K<float>(K, bcx, T, H, w, nullptr, dy, dbcx, dw, nullptr, ws, s);
}

}  // namespace sc
