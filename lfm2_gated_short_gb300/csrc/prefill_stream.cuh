// prefill_stream.cuh -- the TMA-streamed prefill kernel (included by forward.cu,
// whose error word and helpers it shares).
//
// Persistent CTAs (several per SM, as many as fit) each own a balanced range
// of rows [cr0, cr1) of a slice of up to 512 channels. A producer warp streams the rows it needs --
// the range plus the K-1 rows before it (window history) and up to K-2 rows
// after it (the sequence-owner extension) -- through NS shared-memory stages
// with 1-D bulk asynchronous copies (cp.async.bulk). Each stage has a "full"
// mbarrier (the copies' byte count) and an "empty" one (one arrival per
// consumer warp), so the consumer warps (4 channels per thread by default:
// 4 warps for a 512-channel slice) run ahead
// or behind each other freely while up to NS stages of copies are in flight:
// bytes in flight per SM do not depend on registers or occupancy. The
// consumers use packed arithmetic (bf16x2 products, f32x2 multiply-adds) in
// the same operation order as the scalar kernels, so the bits are the same.
//
// Sequence ownership follows the tiled kernel: the CTA whose range holds a
// sequence's first row reads the slot state, writes y for at least the first
// K-1 rows of the sequence (possibly past cr1), and writes the final state
// after its read; other CTAs start that sequence at row s0+K-1 or later and
// take their window history from streamed rows of the same sequence.
//
// This file is a fragment of forward.cu: it is included inside namespace sc,
// after the error word, raise_error(), row_u() and kMaxStagedSeqs; the
// mbarrier and bulk-copy helpers come from tma.cuh.
#pragma once

// Build-time shape of the streamed kernel (defaults are the tuned ones):
// channels per consumer thread, rows per stage for bf16 (fp32 uses half),
// and the number of stages.
#ifndef SC_STREAM_CPT
#define SC_STREAM_CPT 4
#endif
#ifndef SC_STREAM_ROWS
#define SC_STREAM_ROWS 2
#endif
#ifndef SC_STREAM_STAGES
#define SC_STREAM_STAGES 4
#endif
#ifndef SC_STREAM_SLICE
#define SC_STREAM_SLICE 512  // channels per CTA slice
#endif
#ifndef SC_STREAM_MIN_CTAS
#define SC_STREAM_MIN_CTAS 4  // CTAs per SM the register budget is sized for
#endif
#ifndef SC_STREAM_STAGED
#define SC_STREAM_STAGED 512  // sequences whose cu_seqlens / slot ids go to shared memory
#endif

constexpr int kStreamCpt = SC_STREAM_CPT;
constexpr int kStreamSlice = SC_STREAM_SLICE;
constexpr int kStreamStaged = SC_STREAM_STAGED;
constexpr int kStreamCuBytes = ((kStreamStaged + 1) * 4 + 127) / 128 * 128;
constexpr int kStreamHeader = 256 + kStreamCuBytes + kStreamStaged * 4;  // barriers, cu, slots
constexpr int kStreamMinRows = 8;                          // rows per CTA at least
static_assert(kStreamSlice / kStreamCpt + 32 <= 1024, "one CTA holds a slice's consumers");

template <typename T>
struct StreamShape {
    static constexpr int R = sizeof(T) == 2 ? SC_STREAM_ROWS
                                            : (SC_STREAM_ROWS > 1 ? SC_STREAM_ROWS / 2 : 1);
    static constexpr int NS = SC_STREAM_STAGES;
};

template <typename T>
constexpr size_t stream_smem_bytes(int CW) {
    return (size_t)kStreamHeader +
           (size_t)StreamShape<T>::NS * StreamShape<T>::R * 3 * CW * sizeof(T);
}

// HB: a conv bias is given (bias != NULL); the bias-free instance carries no
// bias registers or branches.
template <typename T, int K, bool HB>
__global__ void __launch_bounds__(kStreamSlice / kStreamCpt + 32, SC_STREAM_MIN_CTAS)
    k_prefill_stream(const T *__restrict__ bcx, int64_t T_rows, int H, const T *__restrict__ w,
                     const T *__restrict__ bias, const int32_t *__restrict__ cu, int N,
                     const int32_t *__restrict__ slots, T *__restrict__ pool, int n_slots,
                     T *__restrict__ y, int n_slices, int n_row_ctas) {
    constexpr int CPT = kStreamCpt;
    constexpr int NP = CPT / 2;
    constexpr int R = StreamShape<T>::R;
    constexpr int NS = StreamShape<T>::NS;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + 128);
    int32_t *s_cu = reinterpret_cast<int32_t *>(smem + 256);
    int32_t *s_slot = reinterpret_cast<int32_t *>(smem + 256 + kStreamCuBytes);
    T *stage = reinterpret_cast<T *>(smem + kStreamHeader);

    const int tid = threadIdx.x;
    const int n_consumers = blockDim.x - 32;          // consumer threads; the last warp produces
    const bool producer = tid >= n_consumers;
    const int slice = blockIdx.x % n_slices;
    const int64_t rc = blockIdx.x / n_slices;
    const int c0 = slice * kStreamSlice;
    const int CW = min(kStreamSlice, H);              // stage stride (channels)
    const int cw = min(kStreamSlice, H - c0);         // channels in this slice
    const bool active = !producer && tid * CPT < cw;
    const int h0 = c0 + tid * CPT;
    const int64_t cr0 = rc * T_rows / n_row_ctas, cr1 = (rc + 1) * T_rows / n_row_ctas;
    const int64_t sr0 = max((int64_t)0, cr0 - (K - 1));
    const int64_t sr1 = min(T_rows, cr1 + (K > 2 ? K - 2 : 0));
    const int n_chunks = (int)((sr1 - sr0 + R - 1) / R);
    const uint32_t sec_bytes = (uint32_t)cw * sizeof(T);
    const bool lead = tid == n_consumers;             // lane 0 of the producer warp

    if (lead) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumers / 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // Before the dependency wait: warm L2 with cu_seqlens, the slot ids and, in
    // the first row range, the state of the slot the first row's sequence
    // names. In a model these come from the host or an earlier step, not from
    // the kernel just before, so the loads after the wait hit L2. Hints only:
    // nothing read here is used as a value (see prefetch_l2, slot_hint).
    if (!producer && N <= kStreamStaged) {
        for (int j = tid * 32; j <= N; j += n_consumers * 32) {
            prefetch_l2(cu + j);
            if (j < N) prefetch_l2(slots + j);
        }
        if (cr0 == 0 && active && N > 0) {
            const int hint = slot_hint(slots);
            if (hint >= 0 && hint < n_slots) prefetch_l2(pool + ((int64_t)hint * H + h0) * K);
        }
    }
    pdl_wait();  // everything below may read what earlier kernels in the stream wrote
    pdl_launch_dependents();

    f32x2 wp[K][NP], win[K][NP], bp[NP];
    if (active) {
        load_taps<T, CPT, K>(w + (int64_t)h0 * K, wp);  // in flight during the checks
        if constexpr (HB) {
#pragma unroll
            for (int q = 0; q < NP; ++q)
                bp[q] = f2_make(ld_elem(bias + h0 + 2 * q), ld_elem(bias + h0 + 2 * q + 1));
        }
    }

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
    // Rows depend only on T, so the first stages are requested before cu_seqlens
    // is even read; a bad cu_seqlens then only costs draining them.
    const int first = cr0 < cr1 ? min(NS, n_chunks) : 0;
    if (lead)
        for (int c = 0; c < first; ++c) issue(c);
    auto drain = [&](int from, int to) {  // let this CTA's own copies land before exiting
        for (int c = from; c < to; ++c) mbar_wait_bounded(&full[c % NS], (uint32_t)(c / NS) & 1u);
    };

    const bool staged = N <= kStreamStaged;
    int bad = 0;
    for (int j = tid; j <= N; j += blockDim.x) {
        const int32_t c = gld(cu + j);
        if (staged) {
            s_cu[j] = c;
            if (j < N) s_slot[j] = gld(slots + j);
        }
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && gld(cu + j + 1) < c) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && tid == 0) raise_error(SC_DEV_BAD_SEQLENS);
        if (lead) drain(0, first);
        return;
    }
    if (cr0 >= cr1) return;

    if (producer) {
        if (!lead) return;
        int c = first;
        for (; c < n_chunks; ++c) {
            const uint32_t parity = (uint32_t)(c / NS - 1) & 1u;  // consumers freed use c-NS
            if (!mbar_wait_bounded(&empty[c % NS], parity)) {
                raise_error(SC_DEV_TIMEOUT);
                break;
            }
            issue(c);
        }
        drain(max(0, c - NS), c);
        return;
    }

    auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : gld(cu + j); };
    int lo = 0, hi = N - 1;  // largest i with cu[i] <= sr0: the sequence holding row sr0
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (CU(mid) <= sr0) lo = mid; else hi = mid - 1;
    }
    int i = lo;
    int64_t s0 = CU(i), s1 = CU(i + 1);

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
            const int slot = staged ? s_slot[i] : gld(slots + i);
            ok = slot >= 0 && slot < n_slots;
            if (!ok && owner && slice == 0 && tid == 0) raise_error(SC_DEV_BAD_SLOT);
            if (ok && owner) st = pool + ((int64_t)slot * H + h0) * K;
        }
        if (owner && ok && active) {
            load_taps<T, CPT, K>(st, win);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int q = 0; q < NP; ++q) win[k][q] = 0ull;
        }
    };
    auto finish = [&]() {  // the window now holds the sequence's final state
        if (owner && ok && active) store_taps<T, CPT, K>(st, win);
    };
    // One row: u into the window; y when the row is one of this CTA's outputs.
    auto row_step = [&](uint32_t a, int64_t row, bool out) {
        f32x2 u[NP];
        Pairs<T, CPT>::gate(lds_sec<T, CPT>(a), lds_sec<T, CPT>(a + 2 * CW * sizeof(T)), u);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int k = 0; k + 1 < K; ++k) win[k][q] = win[k + 1][q];
            win[K - 1][q] = u[q];
        }
        if (out) {
            f32x2 cz[NP], yv[NP];
            Pairs<T, CPT>::widen(lds_sec<T, CPT>(a + CW * sizeof(T)), cz);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                f32x2 z = f2_mul(wp[0][q], win[0][q]);
#pragma unroll
                for (int k = 1; k < K; ++k) z = f2_fma(wp[k][q], win[k][q], z);
                if constexpr (HB) z = f2_fma(f2_make(1.f, 1.f), bp[q], z);  // z + b, one rounding
                yv[q] = f2_mul(cz[q], z);
            }
            Pairs<T, CPT>::store(y + row * (int64_t)H + h0, yv);
        }
    };
    enter();

    const int warp_lane = tid & 31;
    const uint32_t stage_addr = smem_addr(stage) + (uint32_t)(tid * CPT * sizeof(T));
    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % NS;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(c / NS) & 1u)) {
            if (warp_lane == 0) raise_error(SC_DEV_TIMEOUT);
            return;  // the producer drains its copies before the CTA exits
        }
        const int64_t rb = sr0 + (int64_t)c * R;
        const uint32_t a0 = stage_addr + (uint32_t)((s * R) * 3 * CW * sizeof(T));
        if (ok && rb >= oa && rb + R <= oe) {
            // Every row of the stage is an output row of one sequence (oe <= s1).
            if (active) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr)
                    row_step(a0 + (uint32_t)(rr * 3 * CW * sizeof(T)), rb + rr, true);
            }
        } else {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const int64_t row = rb + rr;
                if (row >= sr1) break;
                if (row >= s1) {
                    finish();
                    do {
                        ++i;
                        s0 = CU(i);
                        s1 = CU(i + 1);
                    } while (row >= s1);
                    enter();
                }
                if (active)
                    row_step(a0 + (uint32_t)(rr * 3 * CW * sizeof(T)), row,
                             ok && row >= oa && row < oe);
            }
        }
        __syncwarp();
        if (warp_lane == 0) mbar_arrive(&empty[s]);
    }

    if (s1 <= sr1) {
        finish();
    } else if (owner && ok && active) {
        // The sequence continues past this CTA's stream: rebuild its last K values.
        f32x2 f[K][NP];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const T *p = bcx + (s1 - K + k) * 3 * (int64_t)H + h0;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float b0 = ld_elem(p + 2 * q), b1 = ld_elem(p + 2 * q + 1);
                const float x0 = ld_elem(p + 2 * H + 2 * q), x1 = ld_elem(p + 2 * H + 2 * q + 1);
                f[k][q] = f2_make(gate_in<T>(b0, x0), gate_in<T>(b1, x1));
            }
        }
        store_taps<T, CPT, K>(st, f);
    }
}
