// prefill_stream.cuh -- the TMA-streamed prefill kernel (included by forward.cu,
// whose error word and helpers it shares).
//
// One CTA per SM (persistent) owns a balanced range of rows [cr0, cr1) of a
// slice of up to 2048 channels. Thread 0 streams the rows it needs -- the
// range plus the K-1 rows before it (window history) and up to K-2 rows after
// it (the sequence-owner extension) -- through NS shared-memory stages with
// 1-D bulk asynchronous copies (cp.async.bulk) completing on one mbarrier per
// stage; every thread then takes 8 channels of each row from shared memory.
// The copies of the next NS stages are in flight while a stage is computed,
// so bytes in flight per SM do not depend on registers or occupancy.
//
// Sequence ownership follows the tiled kernel: the CTA whose range holds a
// sequence's first row reads the slot state, writes y for at least the first
// K-1 rows of the sequence (possibly past cr1), and writes the final state
// after its read; other CTAs start that sequence at row s0+K-1 or later and
// take their window history from streamed rows of the same sequence.
//
// This file is a fragment of forward.cu: it is included inside namespace sc,
// after the error word, raise_error(), row_u() and kMaxStagedSeqs.
#pragma once

constexpr int kStreamStages = 4;
constexpr int kStreamThreads = 256;                       // 8 channels each
constexpr int kStreamSlice = kStreamThreads * kCh;        // channels per CTA slice
constexpr int kStreamHeader = 128 + ((kMaxStagedSeqs + 1) * 4 + 127) / 128 * 128;
constexpr int kStreamMinRows = 8;                         // rows per CTA at least
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

template <typename T>
struct StreamRows {
    static constexpr int R = sizeof(T) == 2 ? 4 : 2;  // rows per stage (12 / 24 KB per row)
};

template <typename T>
constexpr size_t stream_smem_bytes(int CW) {
    return (size_t)kStreamHeader + (size_t)kStreamStages * StreamRows<T>::R * 3 * CW * sizeof(T);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with this parity to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

template <typename T>
__device__ __forceinline__ void lds_row(const T *p, float (&f)[kCh]) {
    Row<T> r;
#pragma unroll
    for (int i = 0; i < Dt<T>::Q; ++i) r.q[i] = lds128(reinterpret_cast<const uint4 *>(p) + i);
    unpack_row(r, f);
}

template <typename T, int K>
__global__ void __launch_bounds__(kStreamThreads, 1)
    k_prefill_stream(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
                     const int32_t *__restrict__ cu, int N, const int32_t *__restrict__ slots,
                     T *__restrict__ pool, int n_slots, T *__restrict__ y, int n_slices,
                     int n_row_ctas) {
    constexpr int R = StreamRows<T>::R;
    constexpr int NS = kStreamStages;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    int32_t *s_cu = reinterpret_cast<int32_t *>(smem + 128);
    T *stage = reinterpret_cast<T *>(smem + kStreamHeader);

    const int tid = threadIdx.x;
    const int slice = blockIdx.x % n_slices;
    const int64_t rc = blockIdx.x / n_slices;
    const int c0 = slice * kStreamSlice;
    const int CW = min(kStreamSlice, H);          // stage stride (channels)
    const int cw = min(kStreamSlice, H - c0);     // channels in this slice
    const bool active = tid * kCh < cw;
    const int h0 = c0 + tid * kCh;
    const int64_t cr0 = rc * T_rows / n_row_ctas, cr1 = (rc + 1) * T_rows / n_row_ctas;
    const int64_t sr0 = max((int64_t)0, cr0 - (K - 1));
    const int64_t sr1 = min(T_rows, cr1 + (K > 2 ? K - 2 : 0));

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
    }
    const bool staged = N <= kMaxStagedSeqs;
    int bad = 0;
    for (int j = tid; j <= N; j += blockDim.x) {
        const int32_t c = cu[j];
        if (staged) s_cu[j] = c;
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && cu[j + 1] < c) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && tid == 0) raise_error(SC_DEV_BAD_SEQLENS);
        return;
    }
    if (cr0 >= cr1) return;

    const int n_chunks = (int)((sr1 - sr0 + R - 1) / R);
    const uint32_t sec_bytes = (uint32_t)cw * sizeof(T);
    auto issue = [&](int c) {
        const int s = c % NS;
        const int64_t rb = sr0 + (int64_t)c * R;
        const int rows = (int)min((int64_t)R, sr1 - rb);
        mbar_arrive_expect_tx(&full[s], (uint32_t)rows * 3u * sec_bytes);
        for (int rr = 0; rr < rows; ++rr) {
            const T *src = bcx + (rb + rr) * 3 * (int64_t)H + c0;
            T *dst = stage + (size_t)(s * R + rr) * 3 * CW;
#pragma unroll
            for (int q = 0; q < 3; ++q)
                bulk_copy_g2s(dst + (size_t)q * CW, src + (int64_t)q * H, sec_bytes, &full[s]);
        }
    };
    if (tid == 0)
        for (int c = 0; c < min(NS, n_chunks); ++c) issue(c);

    auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : cu[j]; };
    int lo = 0, hi = N - 1;  // largest i with cu[i] <= sr0: the sequence holding row sr0
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (CU(mid) <= sr0) lo = mid; else hi = mid - 1;
    }
    int i = lo;
    int64_t s0 = CU(i), s1 = CU(i + 1);

    float wt[kCh][K], win[kCh][K];
    if (active) load_block<T, K>(w + (int64_t)h0 * K, wt);
    bool owner = false, ok = false;
    int64_t oa = 0, oe = 0;
    T *st = nullptr;

    // Start sequence i at row max(s0, sr0): its output rows here, its slot, its window.
    auto enter = [&]() {
        // Sequences starting in the extension rows past cr1 belong to the next CTA.
        owner = s0 >= cr0 && s0 < cr1;
        if (owner) {
            oa = s0;
            oe = min(s1, max(cr1, s0 + (K - 1)));
        } else {
            oa = max(cr0, s0 + (K - 1));
            oe = min(s1, cr1);
        }
        ok = false;
        if (oa < oe) {
            const int slot = slots[i];
            ok = slot >= 0 && slot < n_slots;
            if (!ok && owner && slice == 0 && tid == 0) raise_error(SC_DEV_BAD_SLOT);
            if (ok && owner) st = pool + ((int64_t)slot * H + h0) * K;
        }
        if (owner && ok && active) {
            load_block<T, K>(st, win);
        } else {
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
                for (int k = 0; k < K; ++k) win[ch][k] = 0.f;
        }
    };
    auto finish = [&]() {  // the window now holds the sequence's final state
        if (owner && ok && active) store_block<T, K>(st, win);
    };
    enter();

    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % NS;
        const bool timed_out = !mbar_wait_bounded(&full[s], (uint32_t)(c / NS) & 1u);
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) {
                raise_error(SC_DEV_TIMEOUT);
                const int issued = min(n_chunks, c + NS);
                for (int cc = c; cc < issued; ++cc)  // let our own copies land before exiting
                    mbar_wait_bounded(&full[cc % NS], (uint32_t)(cc / NS) & 1u);
            }
            return;
        }
        const int64_t rb = sr0 + (int64_t)c * R;
        const int rows = (int)min((int64_t)R, sr1 - rb);
        for (int rr = 0; rr < rows; ++rr) {
            const int64_t row = rb + rr;
            if (row >= s1) {
                finish();
                do {
                    ++i;
                    s0 = CU(i);
                    s1 = CU(i + 1);
                } while (row >= s1);
                enter();
            }
            if (!active) continue;
            const T *p = stage + (size_t)(s * R + rr) * 3 * CW + tid * kCh;
            float b[kCh], x[kCh];
            lds_row(p, b);
            lds_row(p + 2 * CW, x);
            if (ok && row >= oa && row < oe) {
                float cg[kCh], out[kCh];
                lds_row(p + CW, cg);
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch)
                    out[ch] = cg[ch] * slide_dot<K>(win[ch], wt[ch], gate_in<T>(b[ch], x[ch]));
                store_row(y + row * (int64_t)H + h0, out);
            } else {
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) {
                    const float u = gate_in<T>(b[ch], x[ch]);
#pragma unroll
                    for (int k = 0; k + 1 < K; ++k) win[ch][k] = win[ch][k + 1];
                    win[ch][K - 1] = u;
                }
            }
        }
        __syncthreads();  // every thread is done with stage s
        if (tid == 0 && c + NS < n_chunks) issue(c + NS);
    }

    if (s1 <= sr1) {
        finish();
    } else if (owner && ok && active) {
        // The sequence continues past this CTA's stream: rebuild its last K values.
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float u[kCh];
            row_u<T>(bcx, s1 - K + k, H, h0, u);
#pragma unroll
            for (int ch = 0; ch < kCh; ++ch) win[ch][k] = u[ch];
        }
        store_block<T, K>(st, win);
    }
}
