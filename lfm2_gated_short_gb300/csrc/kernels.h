// kernels.h -- internal launchers behind the C ABI (api.cu). Arguments are
// already validated by the caller; these only pick a template instance and
// enqueue on the stream. All return the cudaError_t of the launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sc {

// Prefill: rows_per_thread 0 selects the TMA-streamed kernel (one CTA per SM),
// 4/8/16/32 the register-tiled kernel with that many rows per thread.
// bias (here and below) is the optional per-channel conv bias, NULL for none.
cudaError_t launch_prefill(int dtype, int H, int K, const void *bcx, int64_t T, const void *w,
                           const void *bias, const int32_t *cu_seqlens, int N,
                           const int32_t *slot_ids, void *pool, int n_slots, void *y,
                           int rows_per_thread, int sm_count, cudaStream_t stream);

cudaError_t launch_decode(int dtype, int H, int K, const void *bcx, int N, const void *w,
                          const void *bias, const int32_t *slot_ids, void *pool, int n_slots,
                          void *y, cudaStream_t stream);

cudaError_t launch_verify(int dtype, int H, int K, const void *bcx, int N, int D,
                          const void *w, const void *bias, const int32_t *slot_ids,
                          const void *pool, int n_slots, void *win, void *y,
                          cudaStream_t stream);

// L layers at once: win [L, N, D, H, K], pool [L, n_slots, H, K].
cudaError_t launch_rollback(int dtype, int H, int K, int L, int N, int D, const void *win,
                            const int32_t *accepted, const int32_t *slot_ids, void *pool,
                            int n_slots, cudaStream_t stream);

// Bytes of fp32 partials the backward writes: one H*K dW block per row range,
// plus H dbias entries per row range when dbias is wanted.
size_t backward_partial_bytes(int H, int K, int64_t T, bool with_dbias);
// The caller-workspace size: room for both.
size_t backward_workspace_bytes(int H, int K, int64_t T);

// dbias (fp32 [H]) is written when non-NULL.
cudaError_t launch_backward(int dtype, int H, int K, const void *bcx, int64_t T,
                            const void *w, const void *bias, const void *dy, void *dbcx,
                            float *dw, float *dbias, void *workspace, cudaStream_t stream);

// Packed varlen backward with initial states (NULL: zeros), an optional
// final-state gradient (NULL: zeros) and an optional initial-state gradient
// output (NULL: not written). Same workspace size as launch_backward.
cudaError_t launch_backward_varlen(int dtype, int H, int K, const void *bcx, int64_t T,
                                   const void *w, const void *bias, const int32_t *cu_seqlens,
                                   int N, const void *init, const void *dy,
                                   const float *d_final, void *dbcx, float *dw, float *dbias,
                                   float *d_init, void *workspace, cudaStream_t stream);

// The bias-free backward kernels with their dW partials in the library's
// fixed device scratch (kNoAllocScratchBytes) instead of a caller workspace.
// The caller checks backward_partial_bytes(H, K, T, false) <=
// kNoAllocScratchBytes first.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
cudaError_t launch_backward_noalloc(int dtype, int H, int K, const void *bcx, int64_t T,
                                    const void *w, const void *dy, void *dbcx, float *dw,
                                    cudaStream_t stream);

// The layer's projections (bf16): in_proj fused with the ShortConv, writing y
// and, through k_commit_states, the slots' new states (workspace: the last K
// values of u per sequence, in_proj_workspace_bytes); out_proj a plain GEMM.
size_t in_proj_workspace_bytes(int H, int K, int N);
cudaError_t launch_in_proj_prefill(int D, int H, int K, const void *hidden, int64_t T,
                                   const void *w_in, const void *w, const void *bias,
                                   const int32_t *cu_seqlens, int N, const int32_t *slot_ids,
                                   void *pool, int n_slots, void *y, void *workspace,
                                   int sm_count, cudaStream_t stream);
cudaError_t launch_out_proj(int H, int D, const void *y, int64_t T, const void *w_out, void *out,
                            int sm_count, cudaStream_t stream);
// in_proj fused with the decode of N one-token sequences (bf16): y [N, H] and
// the slots' new states, in one launch.
cudaError_t launch_in_proj_decode(int D, int H, int K, const void *hidden, int N,
                                  const void *w_in, const void *w, const void *bias,
                                  const int32_t *slot_ids, void *pool, int n_slots, void *y,
                                  int sm_count, cudaStream_t stream);
cudaError_t take_error_proj(cudaStream_t stream, unsigned int *code);

// Take (read and clear) the backward translation unit's error word.
cudaError_t take_error_backward(cudaStream_t stream, unsigned int *code);

// Slot pool: claim n_claim free slots (lowest first, all-or-nothing) and
// zero their states when pool != NULL; release slots; copy states.
cudaError_t launch_slots_claim(uint32_t *in_use, int n_slots, int n_claim, int32_t *out,
                               void *pool, int64_t state_bytes, cudaStream_t stream);
cudaError_t launch_slots_release(uint32_t *in_use, int n_slots, const int32_t *slots, int n,
                                 cudaStream_t stream);
cudaError_t launch_pool_copy(const int32_t *src, const int32_t *dst, int n, int64_t state_bytes,
                             void *pool, int n_slots, cudaStream_t stream);
cudaError_t take_error_slots(cudaStream_t stream, unsigned int *code);
// A one-thread kernel whose bounded wait must run out and set SC_DEV_TIMEOUT.
cudaError_t launch_wait_limit_check(cudaStream_t stream);

// Read and clear the device error word of the current device (synchronous
// with respect to `stream`).
cudaError_t read_and_clear_error(cudaStream_t stream, unsigned int *code);

// The bounds-checked build (-DSC_BOUNDS_CHECK): a buffer a call may touch,
// [base, base + bytes), writable or read only. The entry points install the
// call's buffers in the table of each translation unit they launch into.
struct BoundsRegion {
    uint64_t base;
    uint64_t bytes;
    uint32_t writable;
    uint32_t pad;
};
constexpr int kMaxBoundsRegions = 16;
#ifdef SC_BOUNDS_CHECK
enum BoundsUnit { kUnitForward = 0, kUnitBackward = 1, kUnitProj = 2, kUnitSlots = 3 };
cudaError_t bounds_install(int unit, const BoundsRegion *r, int n, cudaStream_t stream);
// The first address any unit refused since the last call (0 when none), cleared.
cudaError_t bounds_take_first_bad(cudaStream_t stream, unsigned long long *addr);
cudaError_t bounds_install_backward(const BoundsRegion *r, int n, cudaStream_t stream);
cudaError_t bounds_install_proj(const BoundsRegion *r, int n, cudaStream_t stream);
cudaError_t bounds_install_slots(const BoundsRegion *r, int n, cudaStream_t stream);
cudaError_t bounds_take_backward(cudaStream_t stream, unsigned long long *addr);
cudaError_t bounds_take_proj(cudaStream_t stream, unsigned long long *addr);
cudaError_t bounds_take_slots(cudaStream_t stream, unsigned long long *addr);
#endif

}  // namespace sc
