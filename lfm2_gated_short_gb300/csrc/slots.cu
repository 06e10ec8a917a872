// slots.cu -- the conv-state slot pool on the device: claim, release, copy.
//
// The MAX LFM2 article ("MAX Pipelines 的 LFM2 架构支持", section "推理状态管理：
// ConvStateCache 与卷积状态生命周期") keeps one conv state per request slot:
// a request claims a free slot (an error when none is free), starts from a
// zero state and releases the slot when done. Here the in-use set is a
// caller-owned device bitmap, so a serving loop can claim and release slots
// in stream order without a host round trip. Copying a slot's state to
// another slot (a snapshot) lets a shared prefix's state be reused.
#include "common.cuh"
#include "errors.cuh"
#include "kernels.h"
#include "launch.h"
#include "shortconv.h"
#include "tma.cuh"

namespace sc {

constexpr int kClaimThreads = 1024;

// One CTA: thread t owns a contiguous run of bitmap words and counts its free
// slots; an exclusive scan over threads ranks every free slot; the n_claim
// lowest-ranked ones are taken in increasing slot order. All-or-nothing.
__global__ void __launch_bounds__(kClaimThreads)
    k_slots_claim(uint32_t *__restrict__ in_use, int n_slots, int n_claim,
                  int32_t *__restrict__ out) {
    __shared__ int s_scan[kClaimThreads];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int n_words = (n_slots + 31) / 32;
    const int per = (n_words + kClaimThreads - 1) / kClaimThreads;
    const int w0 = min(n_words, tid * per), w1 = min(n_words, w0 + per);
    auto valid = [&](int wi) -> uint32_t {  // bits of word wi that are real slots
        const int rem = n_slots - wi * 32;
        return rem >= 32 ? 0xFFFFFFFFu : ((1u << rem) - 1u);
    };
    int mine = 0;
    for (int wi = w0; wi < w1; ++wi) mine += __popc(~gld(in_use + wi) & valid(wi));
    s_scan[tid] = mine;
    __syncthreads();
    for (int off = 1; off < kClaimThreads; off <<= 1) {  // inclusive scan (Hillis-Steele)
        const int v = tid >= off ? s_scan[tid - off] : 0;
        __syncthreads();
        s_scan[tid] += v;
        __syncthreads();
    }
    const int total = s_scan[kClaimThreads - 1];
    if (total < n_claim) {
        for (int i = tid; i < n_claim; i += kClaimThreads) gst(out + i, -1);
        if (tid == 0) raise_error(SC_DEV_NO_SLOT);
        return;
    }
    int rank = s_scan[tid] - mine;  // free slots before this thread's words
    for (int wi = w0; wi < w1 && rank < n_claim; ++wi) {
        uint32_t word = gld(in_use + wi);
        uint32_t fr = ~word & valid(wi);
        while (fr != 0u && rank < n_claim) {
            const int b = __ffs(fr) - 1;
            fr &= fr - 1u;
            word |= 1u << b;
            gst(out + rank++, wi * 32 + b);
        }
        gst(in_use + wi, word);
    }
}

// Zero the states of the slots just claimed (fresh sequences start from zero).
__global__ void __launch_bounds__(256)
    k_slots_zero(const int32_t *__restrict__ slots, int n, int64_t q_per_slot,
                 uint4 *__restrict__ pool, int n_slots) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (unit >= (int64_t)n * q_per_slot) return;
    const int s = gld(slots + unit / q_per_slot);
    if (s < 0 || s >= n_slots) return;  // nothing was claimed
    gst(pool + (int64_t)s * q_per_slot + unit % q_per_slot, make_uint4(0u, 0u, 0u, 0u));
}

__global__ void __launch_bounds__(256)
    k_slots_release(uint32_t *__restrict__ in_use, int n_slots,
                    const int32_t *__restrict__ slots, int n) {
    pdl_wait();
    pdl_launch_dependents();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int s = gld(slots + i);
    if (s < 0 || s >= n_slots) {
        raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    const uint32_t bit = 1u << (s & 31);
    if (!SC_WR_OK(in_use + (s >> 5), 4)) return;
    const uint32_t old = atomicAnd(&in_use[s >> 5], ~bit);
    if (!(old & bit)) raise_error(SC_DEV_BAD_SLOT);  // it was not in use
}

__global__ void __launch_bounds__(256)
    k_pool_copy(const int32_t *__restrict__ src, const int32_t *__restrict__ dst, int n,
                int64_t q_per_slot, uint4 *__restrict__ pool, int n_slots) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (unit >= (int64_t)n * q_per_slot) return;
    const int i = (int)(unit / q_per_slot);
    const int64_t q = unit % q_per_slot;
    const int s = gld(src + i), d = gld(dst + i);
    if (s < 0 || s >= n_slots || d < 0 || d >= n_slots) {
        if (q == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    gst(pool + (int64_t)d * q_per_slot + q, gld(pool + (int64_t)s * q_per_slot + q));
}

cudaError_t launch_slots_claim(uint32_t *in_use, int n_slots, int n_claim, int32_t *out,
                               void *pool, int64_t state_bytes, cudaStream_t stream) {
    cudaError_t e = launch_pdl(k_slots_claim, dim3(1), dim3(kClaimThreads), 0, stream, in_use,
                               n_slots, n_claim, out);
    if (e != cudaSuccess || pool == nullptr || n_claim == 0) return e;
    const int64_t q = state_bytes / 16;
    const int64_t blocks = ((int64_t)n_claim * q + 255) / 256;
    return launch_pdl(k_slots_zero, dim3((unsigned)blocks), dim3(256), 0, stream,
                      (const int32_t *)out, n_claim, q, (uint4 *)pool, n_slots);
}

cudaError_t launch_slots_release(uint32_t *in_use, int n_slots, const int32_t *slots, int n,
                                 cudaStream_t stream) {
    return launch_pdl(k_slots_release, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream,
                      in_use, n_slots, slots, n);
}

cudaError_t launch_pool_copy(const int32_t *src, const int32_t *dst, int n, int64_t state_bytes,
                             void *pool, int n_slots, cudaStream_t stream) {
    const int64_t q = state_bytes / 16;
    const int64_t blocks = ((int64_t)n * q + 255) / 256;
    return launch_pdl(k_pool_copy, dim3((unsigned)blocks), dim3(256), 0, stream, src, dst, n, q,
                      (uint4 *)pool, n_slots);
}

// ------------------------------------------------------- wait-limit check
//
// Every kernel here that waits on an mbarrier (the streamed prefill and
// backwards, the projections) gives up after kWaitLimitNs, sets
// SC_DEV_TIMEOUT and returns instead of hanging. This one-thread kernel waits
// with that same bounded wait on a barrier that nothing ever completes, so
// the give-up and the report can be checked on a device without any copy
// failing.
__global__ void k_wait_limit_check() {
    __shared__ uint64_t bar;
    pdl_wait();
    pdl_launch_dependents();
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (!mbar_wait_bounded(&bar, 0u)) raise_error(SC_DEV_TIMEOUT);
}

cudaError_t launch_wait_limit_check(cudaStream_t stream) {
    return launch_pdl(k_wait_limit_check, dim3(1), dim3(1), 0, stream);
}

cudaError_t take_error_slots(cudaStream_t stream, unsigned int *code) {
    return take_error_here(stream, code);
}

#ifdef SC_BOUNDS_CHECK
cudaError_t bounds_install_slots(const BoundsRegion *r, int n, cudaStream_t stream) {
    return bounds_install_here(r, n, stream);
}
cudaError_t bounds_take_slots(cudaStream_t stream, unsigned long long *addr) {
    return bounds_take_first_bad_here(stream, addr);
}
#endif

}  // namespace sc
