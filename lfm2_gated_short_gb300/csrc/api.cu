// api.cu -- the extern "C" entry points declared in include/shortconv.h.
//
// Each entry point validates its arguments on the host (no CUDA call before
// the arguments are known good), then enqueues the kernel(s) on the caller's
// stream. Nothing is allocated and nothing is synchronized, except in
// shortconv_get_error.
#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "kernels.h"
#include "shortconv.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// A pointer describing `bytes` bytes: NULL allowed only when empty.
bool ptr_ok(const void *p, size_t bytes, uintptr_t align) {
    if (bytes == 0) return p == nullptr || aligned(p, align);
    return p != nullptr && aligned(p, align);
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (na == 0 || nb == 0 || a == nullptr || b == nullptr) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t elem_size(sc_dtype d) { return d == SC_BF16 ? 2 : 4; }

// An optional array: NULL (absent) or aligned.
bool opt_ok(const void *p, uintptr_t align) { return p == nullptr || aligned(p, align); }

// Common size checks: dtype, H, K.
sc_status check_shape(sc_dtype dtype, int H, int K) {
    if (dtype != SC_F32 && dtype != SC_BF16) return SC_EUNSUPPORTED;
    if (H <= 0 || K <= 0) return SC_EINVAL;
    if (H % 8 != 0 || K > 4) return SC_EUNSUPPORTED;
    if ((int64_t)H * 3 > INT32_MAX / 2) return SC_EUNSUPPORTED;
    return SC_OK;
}

int sm_count_of_current_device() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

sc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SC_OK : SC_ECUDA; }

#ifdef SC_BOUNDS_CHECK
// The bounds-checked build: before its launches, each entry point installs
// the buffers the call may read (RO) and write (RW), in the order listed at
// the call, in the table of the translation unit it launches into.
// shortconv_bounds_trim_next shortens one listed buffer of the next call.
std::mutex g_trim_mu;
int g_trim_index = -1;
uint64_t g_trim_bytes = 0;

sc::BoundsRegion RO(const void *p, size_t bytes) {
    return sc::BoundsRegion{reinterpret_cast<uint64_t>(p), p ? (uint64_t)bytes : 0, 0, 0};
}
sc::BoundsRegion RW(void *p, size_t bytes) {
    return sc::BoundsRegion{reinterpret_cast<uint64_t>(p), p ? (uint64_t)bytes : 0, 1, 0};
}
sc_status bounds_install(int unit, std::initializer_list<sc::BoundsRegion> regions,
                         void *stream) {
    sc::BoundsRegion r[sc::kMaxBoundsRegions];
    int n = 0;
    for (const sc::BoundsRegion &x : regions) {
        if (n == sc::kMaxBoundsRegions) return SC_EUNSUPPORTED;
        r[n++] = x;
    }
    {
        std::lock_guard<std::mutex> lock(g_trim_mu);
        if (g_trim_index >= 0 && g_trim_index < n) {
            uint64_t &b = r[g_trim_index].bytes;
            b = b > g_trim_bytes ? b - g_trim_bytes : 0;
        }
        g_trim_index = -1;
        g_trim_bytes = 0;
    }
    return from_cuda(sc::bounds_install(unit, r, n, (cudaStream_t)stream));
}
#define SC_BOUNDS_INSTALL(unit, ...)                                           \
    do {                                                                      \
        const sc_status bst = bounds_install(sc::unit, {__VA_ARGS__}, stream); \
        if (bst != SC_OK) return bst;                                         \
    } while (0)
#else
#define SC_BOUNDS_INSTALL(unit, ...) \
    do {                             \
    } while (0)
#endif

sc_status prefill_impl(sc_dtype dtype, int H, int K, const void *bcx, int64_t T, const void *w,
                       const void *bias, const int32_t *cu_seqlens, int N,
                       const int32_t *slot_ids, void *pool, int n_slots, void *y,
                       int rows_per_thread, void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (T < 0 || T > INT32_MAX || N < 0 || n_slots <= 0) return SC_EINVAL;
    if (N == 0 && T != 0) return SC_EINVAL;
    if (rows_per_thread != 0 && rows_per_thread != 4 && rows_per_thread != 8 &&
        rows_per_thread != 16 && rows_per_thread != 32)
        return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t n_bcx = (size_t)T * 3 * H * es, n_y = (size_t)T * H * es;
    const size_t n_w = (size_t)H * K * es, n_pool = (size_t)n_slots * H * K * es;
    const size_t n_b = bias ? (size_t)H * es : 0;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(y, n_y, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(pool, n_pool, 16) || !ptr_ok(cu_seqlens, (size_t)(N + 1) * 4, 4) ||
        !ptr_ok(slot_ids, (size_t)N * 4, 4) || !opt_ok(bias, 16))
        return SC_EINVAL;
    if (overlaps(y, n_y, bcx, n_bcx) || overlaps(y, n_y, pool, n_pool) ||
        overlaps(y, n_y, w, n_w) || overlaps(pool, n_pool, bcx, n_bcx) ||
        overlaps(pool, n_pool, w, n_w) || overlaps(y, n_y, bias, n_b) ||
        overlaps(pool, n_pool, bias, n_b))
        return SC_EINVAL;
    if (N == 0) return SC_OK;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return SC_ECUDA;
    SC_BOUNDS_INSTALL(kUnitForward, RO(bcx, n_bcx), RO(w, n_w), RO(bias, n_b),
                      RO(cu_seqlens, (size_t)(N + 1) * 4), RO(slot_ids, (size_t)N * 4),
                      RW(pool, n_pool), RW(y, n_y));
    return from_cuda(sc::launch_prefill(dtype, H, K, bcx, T, w, bias, cu_seqlens, N, slot_ids,
                                        pool, n_slots, y, rows_per_thread, sms,
                                        (cudaStream_t)stream));
}

}  // namespace

extern "C" {

sc_status shortconv_prefill(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                            const void *w, const void *bias, const int32_t *cu_seqlens, int N,
                            const int32_t *slot_ids, void *pool, int n_slots, void *y,
                            void *stream) {
    return prefill_impl(dtype, H, K, bcx, T, w, bias, cu_seqlens, N, slot_ids, pool, n_slots, y,
                        0, stream);
}

sc_status shortconv_prefill_tiled(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                  const void *w, const void *bias, const int32_t *cu_seqlens,
                                  int N, const int32_t *slot_ids, void *pool, int n_slots,
                                  void *y, int rows_per_thread, void *stream) {
    return prefill_impl(dtype, H, K, bcx, T, w, bias, cu_seqlens, N, slot_ids, pool, n_slots, y,
                        rows_per_thread, stream);
}

sc_status shortconv_decode(sc_dtype dtype, int H, int K, const void *bcx, int N, const void *w,
                           const void *bias, const int32_t *slot_ids, void *pool, int n_slots,
                           void *y, void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (N < 0 || n_slots <= 0) return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t n_bcx = (size_t)N * 3 * H * es, n_y = (size_t)N * H * es;
    const size_t n_w = (size_t)H * K * es, n_pool = (size_t)n_slots * H * K * es;
    const size_t n_b = bias ? (size_t)H * es : 0;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(y, n_y, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(pool, n_pool, 16) || !ptr_ok(slot_ids, (size_t)N * 4, 4) || !opt_ok(bias, 16))
        return SC_EINVAL;
    if (overlaps(y, n_y, bcx, n_bcx) || overlaps(y, n_y, pool, n_pool) ||
        overlaps(y, n_y, w, n_w) || overlaps(pool, n_pool, bcx, n_bcx) ||
        overlaps(pool, n_pool, w, n_w) || overlaps(y, n_y, bias, n_b) ||
        overlaps(pool, n_pool, bias, n_b))
        return SC_EINVAL;
    if (N == 0) return SC_OK;
    SC_BOUNDS_INSTALL(kUnitForward, RO(bcx, n_bcx), RO(w, n_w), RO(bias, n_b),
                      RO(slot_ids, (size_t)N * 4), RW(pool, n_pool), RW(y, n_y));
    return from_cuda(sc::launch_decode(dtype, H, K, bcx, N, w, bias, slot_ids, pool, n_slots, y,
                                       (cudaStream_t)stream));
}

sc_status shortconv_verify(sc_dtype dtype, int H, int K, const void *bcx, int N, int D,
                           const void *w, const void *bias, const int32_t *slot_ids,
                           const void *pool, int n_slots, void *win, void *y, void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (N < 0 || D <= 0 || n_slots <= 0) return SC_EINVAL;
    if ((int64_t)N * D > INT32_MAX) return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t rows = (size_t)N * D;
    const size_t n_bcx = rows * 3 * H * es, n_y = rows * H * es, n_win = rows * H * K * es;
    const size_t n_w = (size_t)H * K * es, n_pool = (size_t)n_slots * H * K * es;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(y, n_y, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(pool, n_pool, 16) || !ptr_ok(win, n_win, 16) ||
        !ptr_ok(slot_ids, (size_t)N * 4, 4) || !opt_ok(bias, 16))
        return SC_EINVAL;
    const void *ins[4] = {bcx, w, pool, bias};
    const size_t nins[4] = {n_bcx, n_w, n_pool, bias ? (size_t)H * es : 0};
    for (int i = 0; i < 4; ++i)
        if (overlaps(y, n_y, ins[i], nins[i]) || overlaps(win, n_win, ins[i], nins[i]))
            return SC_EINVAL;
    if (overlaps(y, n_y, win, n_win)) return SC_EINVAL;
    if (N == 0) return SC_OK;
    SC_BOUNDS_INSTALL(kUnitForward, RO(bcx, n_bcx), RO(w, n_w), RO(bias, nins[3]),
                      RO(slot_ids, (size_t)N * 4), RO(pool, n_pool), RW(win, n_win), RW(y, n_y));
    return from_cuda(sc::launch_verify(dtype, H, K, bcx, N, D, w, bias, slot_ids, pool, n_slots,
                                       win, y, (cudaStream_t)stream));
}

sc_status shortconv_rollback_layers(sc_dtype dtype, int H, int K, int L, int N, int D,
                                   const void *win, const int32_t *accepted,
                                   const int32_t *slot_ids, void *pool, int n_slots,
                                   void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (L <= 0 || N < 0 || D <= 0 || n_slots <= 0) return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t n_win = (size_t)L * N * D * H * K * es;
    const size_t n_pool = (size_t)L * n_slots * H * K * es;
    if (!ptr_ok(win, n_win, 16) || !ptr_ok(pool, n_pool, 16) ||
        !ptr_ok(accepted, (size_t)N * 4, 4) || !ptr_ok(slot_ids, (size_t)N * 4, 4))
        return SC_EINVAL;
    if (overlaps(pool, n_pool, win, n_win) || overlaps(pool, n_pool, accepted, (size_t)N * 4) ||
        overlaps(pool, n_pool, slot_ids, (size_t)N * 4))
        return SC_EINVAL;
    if (N == 0) return SC_OK;
    SC_BOUNDS_INSTALL(kUnitForward, RO(win, n_win), RO(accepted, (size_t)N * 4),
                      RO(slot_ids, (size_t)N * 4), RW(pool, n_pool));
    return from_cuda(sc::launch_rollback(dtype, H, K, L, N, D, win, accepted, slot_ids, pool,
                                         n_slots, (cudaStream_t)stream));
}

sc_status shortconv_rollback(sc_dtype dtype, int H, int K, int N, int D, const void *win,
                             const int32_t *accepted, const int32_t *slot_ids, void *pool,
                             int n_slots, void *stream) {
    return shortconv_rollback_layers(dtype, H, K, 1, N, D, win, accepted, slot_ids, pool,
                                     n_slots, stream);
}

size_t shortconv_backward_workspace_bytes(int H, int K, int64_t T) {
    if (H <= 0 || H % 8 != 0 || K <= 0 || K > 4 || T < 0 || T > INT32_MAX) return 0;
    return sc::backward_workspace_bytes(H, K, T);
}

sc_status shortconv_backward(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                             const void *w, const void *bias, const void *dy, void *dbcx,
                             float *dw, float *dbias, void *workspace, size_t workspace_bytes,
                             void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (T < 0 || T > INT32_MAX) return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t n_bcx = (size_t)T * 3 * H * es, n_dy = (size_t)T * H * es;
    const size_t n_w = (size_t)H * K * es, n_dw = (size_t)H * K * 4;
    const size_t need = sc::backward_workspace_bytes(H, K, T);
    if (workspace_bytes < need) return SC_EINVAL;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(dy, n_dy, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(dbcx, n_bcx, 16) || !ptr_ok(dw, n_dw, 4) || !ptr_ok(workspace, need, 16) ||
        !opt_ok(bias, 16) || !opt_ok(dbias, 4))
        return SC_EINVAL;
    const void *ins[4] = {bcx, w, dy, bias};
    const size_t nins[4] = {n_bcx, n_w, n_dy, bias ? (size_t)H * es : 0};
    const void *outs[4] = {dbcx, dw, dbias, workspace};
    const size_t nouts[4] = {n_bcx, n_dw, dbias ? (size_t)H * 4 : 0, need};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 4; ++i)
            if (overlaps(outs[o], nouts[o], ins[i], nins[i])) return SC_EINVAL;
        for (int p = o + 1; p < 4; ++p)
            if (overlaps(outs[o], nouts[o], outs[p], nouts[p])) return SC_EINVAL;
    }
    SC_BOUNDS_INSTALL(kUnitBackward, RO(bcx, n_bcx), RO(w, n_w), RO(bias, nins[3]),
                      RO(dy, n_dy), RW(dbcx, n_bcx), RW(dw, n_dw), RW(dbias, nouts[2]),
                      RW(workspace, need));
    return from_cuda(sc::launch_backward(dtype, H, K, bcx, T, w, bias, dy, dbcx, dw, dbias,
                                         workspace, (cudaStream_t)stream));
}

sc_status shortconv_backward_varlen(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                    const void *w, const void *bias, const int32_t *cu_seqlens,
                                    int N, const void *init_states, const void *dy,
                                    const float *d_final, void *dbcx, float *dw, float *dbias,
                                    float *d_init, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (T < 0 || T > INT32_MAX || N < 0) return SC_EINVAL;
    if (N == 0 && T != 0) return SC_EINVAL;
    const size_t es = elem_size(dtype);
    const size_t n_bcx = (size_t)T * 3 * H * es, n_dy = (size_t)T * H * es;
    const size_t n_w = (size_t)H * K * es, n_dw = (size_t)H * K * 4;
    const size_t n_st = (size_t)N * H * K * es, n_sf = (size_t)N * H * K * 4;
    const size_t need = sc::backward_workspace_bytes(H, K, T);
    if (workspace_bytes < need) return SC_EINVAL;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(dy, n_dy, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(dbcx, n_bcx, 16) || !ptr_ok(dw, n_dw, 4) || !ptr_ok(workspace, need, 16) ||
        !ptr_ok(cu_seqlens, (size_t)(N + 1) * 4, 4))
        return SC_EINVAL;
    if (!opt_ok(init_states, 4) || !opt_ok(d_final, 4) || !opt_ok(d_init, 4) ||
        !opt_ok(bias, 16) || !opt_ok(dbias, 4))
        return SC_EINVAL;
    const void *ins[7] = {bcx, w, dy, init_states, d_final, cu_seqlens, bias};
    const size_t nins[7] = {n_bcx, n_w, n_dy, init_states ? n_st : 0, d_final ? n_sf : 0,
                            (size_t)(N + 1) * 4, bias ? (size_t)H * es : 0};
    const void *outs[5] = {dbcx, dw, d_init, workspace, dbias};
    const size_t nouts[5] = {n_bcx, n_dw, d_init ? n_sf : 0, need, dbias ? (size_t)H * 4 : 0};
    for (int o = 0; o < 5; ++o) {
        for (int i = 0; i < 7; ++i)
            if (overlaps(outs[o], nouts[o], ins[i], nins[i])) return SC_EINVAL;
        for (int p = o + 1; p < 5; ++p)
            if (overlaps(outs[o], nouts[o], outs[p], nouts[p])) return SC_EINVAL;
    }
    SC_BOUNDS_INSTALL(kUnitBackward, RO(bcx, n_bcx), RO(w, n_w), RO(bias, nins[6]),
                      RO(cu_seqlens, nins[5]), RO(init_states, nins[3]), RO(dy, n_dy),
                      RO(d_final, nins[4]), RW(dbcx, n_bcx), RW(dw, n_dw), RW(dbias, nouts[4]),
                      RW(d_init, nouts[2]), RW(workspace, need));
    return from_cuda(sc::launch_backward_varlen(dtype, H, K, bcx, T, w, bias, cu_seqlens, N,
                                                init_states, dy, d_final, dbcx, dw, dbias,
                                                d_init, workspace, (cudaStream_t)stream));
}

sc_status shortconv_backward_noalloc(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                     const void *w, const void *dy, void *dbcx, float *dw,
                                     void *stream) {
    sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (T < 0 || T > INT32_MAX) return SC_EINVAL;
    if (sc::backward_partial_bytes(H, K, T, false) > sc::kNoAllocScratchBytes)
        return SC_EUNSUPPORTED;
    const size_t es = elem_size(dtype);
    const size_t n_bcx = (size_t)T * 3 * H * es, n_dy = (size_t)T * H * es;
    const size_t n_w = (size_t)H * K * es, n_dw = (size_t)H * K * 4;
    if (!ptr_ok(bcx, n_bcx, 16) || !ptr_ok(dy, n_dy, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(dbcx, n_bcx, 16) || !ptr_ok(dw, n_dw, 4))
        return SC_EINVAL;
    const void *ins[3] = {bcx, w, dy};
    const size_t nins[3] = {n_bcx, n_w, n_dy};
    for (int i = 0; i < 3; ++i)
        if (overlaps(dbcx, n_bcx, ins[i], nins[i]) || overlaps(dw, n_dw, ins[i], nins[i]))
            return SC_EINVAL;
    if (overlaps(dbcx, n_bcx, dw, n_dw)) return SC_EINVAL;
    SC_BOUNDS_INSTALL(kUnitBackward, RO(bcx, n_bcx), RO(w, n_w), RO(dy, n_dy), RW(dbcx, n_bcx),
                      RW(dw, n_dw));  // the launcher adds the fixed scratch array
    return from_cuda(sc::launch_backward_noalloc(dtype, H, K, bcx, T, w, dy, dbcx, dw,
                                                 (cudaStream_t)stream));
}

size_t shortconv_in_proj_workspace_bytes(int H, int K, int N) {
    if (H <= 0 || H % 64 != 0 || K <= 0 || K > 4 || N < 0) return 0;
    return sc::in_proj_workspace_bytes(H, K, N);
}

sc_status shortconv_in_proj_prefill(sc_dtype dtype, int D, int H, int K, const void *hidden,
                                    int64_t T, const void *w_in, const void *w, const void *bias,
                                    const int32_t *cu_seqlens, int N, const int32_t *slot_ids,
                                    void *pool, int n_slots, void *y, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    if (dtype != SC_BF16 && dtype != SC_F32) return SC_EUNSUPPORTED;
    if (D <= 0 || H <= 0 || K <= 0) return SC_EINVAL;
    if (dtype != SC_BF16 || D % 64 != 0 || H % 64 != 0 || K > 4) return SC_EUNSUPPORTED;
    if ((int64_t)H * 3 > INT32_MAX / 2 || D > INT32_MAX / 2) return SC_EUNSUPPORTED;
    if (T < 0 || T > INT32_MAX || N < 0 || n_slots <= 0) return SC_EINVAL;
    if (N == 0 && T != 0) return SC_EINVAL;
    const size_t n_h = (size_t)T * D * 2, n_win = (size_t)3 * H * D * 2, n_w = (size_t)H * K * 2;
    const size_t n_y = (size_t)T * H * 2, n_pool = (size_t)n_slots * H * K * 2;
    const size_t need = sc::in_proj_workspace_bytes(H, K, N);
    if (workspace_bytes < need) return SC_EINVAL;
    if (!ptr_ok(hidden, n_h, 16) || !ptr_ok(w_in, n_win, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(y, n_y, 16) || !ptr_ok(pool, n_pool, 16) || !ptr_ok(workspace, need, 16) ||
        !ptr_ok(cu_seqlens, (size_t)(N + 1) * 4, 4) || !ptr_ok(slot_ids, (size_t)N * 4, 4) ||
        !opt_ok(bias, 16))
        return SC_EINVAL;
    const void *ins[6] = {hidden, w_in, w, bias, cu_seqlens, slot_ids};
    const size_t nins[6] = {n_h, n_win, n_w, bias ? (size_t)H * 2 : 0, (size_t)(N + 1) * 4,
                            (size_t)N * 4};
    const void *outs[3] = {y, pool, workspace};
    const size_t nouts[3] = {n_y, n_pool, need};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(outs[o], nouts[o], ins[i], nins[i])) return SC_EINVAL;
        for (int p = o + 1; p < 3; ++p)
            if (overlaps(outs[o], nouts[o], outs[p], nouts[p])) return SC_EINVAL;
    }
    if (N == 0) return SC_OK;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return SC_ECUDA;
    SC_BOUNDS_INSTALL(kUnitProj, RO(hidden, n_h), RO(w_in, n_win), RO(w, n_w), RO(bias, nins[3]),
                      RO(cu_seqlens, nins[4]), RO(slot_ids, nins[5]), RW(pool, n_pool),
                      RW(y, n_y), RW(workspace, need));
    return from_cuda(sc::launch_in_proj_prefill(D, H, K, hidden, T, w_in, w, bias, cu_seqlens, N,
                                                slot_ids, pool, n_slots, y, workspace, sms,
                                                (cudaStream_t)stream));
}

sc_status shortconv_in_proj_decode(sc_dtype dtype, int D, int H, int K, const void *hidden,
                                   int N, const void *w_in, const void *w, const void *bias,
                                   const int32_t *slot_ids, void *pool, int n_slots, void *y,
                                   void *stream) {
    if (dtype != SC_BF16 && dtype != SC_F32) return SC_EUNSUPPORTED;
    if (D <= 0 || H <= 0 || K <= 0) return SC_EINVAL;
    if (dtype != SC_BF16 || D % 64 != 0 || H % 64 != 0 || K > 4) return SC_EUNSUPPORTED;
    if ((int64_t)H * 3 > INT32_MAX / 2 || D > INT32_MAX / 2) return SC_EUNSUPPORTED;
    if (N < 0 || n_slots <= 0) return SC_EINVAL;
    const size_t n_h = (size_t)N * D * 2, n_win = (size_t)3 * H * D * 2, n_w = (size_t)H * K * 2;
    const size_t n_y = (size_t)N * H * 2, n_pool = (size_t)n_slots * H * K * 2;
    const size_t n_b = bias ? (size_t)H * 2 : 0;
    if (!ptr_ok(hidden, n_h, 16) || !ptr_ok(w_in, n_win, 16) || !ptr_ok(w, n_w, 16) ||
        !ptr_ok(y, n_y, 16) || !ptr_ok(pool, n_pool, 16) || !ptr_ok(slot_ids, (size_t)N * 4, 4) ||
        !opt_ok(bias, 16))
        return SC_EINVAL;
    const void *ins[5] = {hidden, w_in, w, bias, slot_ids};
    const size_t nins[5] = {n_h, n_win, n_w, n_b, (size_t)N * 4};
    const void *outs[2] = {y, pool};
    const size_t nouts[2] = {n_y, n_pool};
    for (int o = 0; o < 2; ++o)
        for (int i = 0; i < 5; ++i)
            if (overlaps(outs[o], nouts[o], ins[i], nins[i])) return SC_EINVAL;
    if (overlaps(y, n_y, pool, n_pool)) return SC_EINVAL;
    if (N == 0) return SC_OK;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return SC_ECUDA;
    SC_BOUNDS_INSTALL(kUnitProj, RO(hidden, n_h), RO(w_in, n_win), RO(w, n_w), RO(bias, n_b),
                      RO(slot_ids, (size_t)N * 4), RW(pool, n_pool), RW(y, n_y));
    return from_cuda(sc::launch_in_proj_decode(D, H, K, hidden, N, w_in, w, bias, slot_ids, pool,
                                               n_slots, y, sms, (cudaStream_t)stream));
}

sc_status shortconv_out_proj(sc_dtype dtype, int H, int D, const void *y, int64_t T,
                             const void *w_out, void *out, void *stream) {
    if (dtype != SC_BF16 && dtype != SC_F32) return SC_EUNSUPPORTED;
    if (D <= 0 || H <= 0) return SC_EINVAL;
    if (dtype != SC_BF16 || H % 64 != 0 || D % 256 != 0) return SC_EUNSUPPORTED;
    if (H > INT32_MAX / 2 || D > INT32_MAX / 2) return SC_EUNSUPPORTED;
    if (T < 0 || T > INT32_MAX) return SC_EINVAL;
    const size_t n_y = (size_t)T * H * 2, n_wo = (size_t)D * H * 2, n_out = (size_t)T * D * 2;
    if (!ptr_ok(y, n_y, 16) || !ptr_ok(w_out, n_wo, 16) || !ptr_ok(out, n_out, 16))
        return SC_EINVAL;
    if (overlaps(out, n_out, y, n_y) || overlaps(out, n_out, w_out, n_wo)) return SC_EINVAL;
    if (T == 0) return SC_OK;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return SC_ECUDA;
    SC_BOUNDS_INSTALL(kUnitProj, RO(y, n_y), RO(w_out, n_wo), RW(out, n_out));
    return from_cuda(sc::launch_out_proj(H, D, y, T, w_out, out, sms, (cudaStream_t)stream));
}

sc_status shortconv_slots_claim(uint32_t *in_use, int n_slots, int n_claim, int32_t *slots_out,
                                sc_dtype dtype, int H, int K, void *pool, void *stream) {
    if (n_slots <= 0 || n_claim < 0 || n_claim > n_slots) return SC_EINVAL;
    const size_t n_bm = (size_t)(n_slots + 31) / 32 * 4;
    if (!ptr_ok(in_use, n_bm, 4) || !ptr_ok(slots_out, (size_t)n_claim * 4, 4)) return SC_EINVAL;
    size_t n_pool = 0;
    int64_t state_bytes = 0;
    if (pool != nullptr) {
        const sc_status st = check_shape(dtype, H, K);
        if (st != SC_OK) return st;
        state_bytes = (int64_t)H * K * elem_size(dtype);
        n_pool = (size_t)n_slots * state_bytes;
        if (!aligned(pool, 16)) return SC_EINVAL;
    }
    if (overlaps(in_use, n_bm, slots_out, (size_t)n_claim * 4) ||
        overlaps(in_use, n_bm, pool, n_pool) || overlaps(slots_out, (size_t)n_claim * 4, pool, n_pool))
        return SC_EINVAL;
    SC_BOUNDS_INSTALL(kUnitSlots, RW(in_use, n_bm), RW(slots_out, (size_t)n_claim * 4),
                      RW(pool, n_pool));
    return from_cuda(sc::launch_slots_claim(in_use, n_slots, n_claim, slots_out, pool,
                                            state_bytes, (cudaStream_t)stream));
}

sc_status shortconv_slots_release(uint32_t *in_use, int n_slots, const int32_t *slot_ids, int n,
                                  void *stream) {
    if (n_slots <= 0 || n < 0) return SC_EINVAL;
    const size_t n_bm = (size_t)(n_slots + 31) / 32 * 4;
    if (!ptr_ok(in_use, n_bm, 4) || !ptr_ok(slot_ids, (size_t)n * 4, 4)) return SC_EINVAL;
    if (overlaps(in_use, n_bm, slot_ids, (size_t)n * 4)) return SC_EINVAL;
    if (n == 0) return SC_OK;
    SC_BOUNDS_INSTALL(kUnitSlots, RW(in_use, n_bm), RO(slot_ids, (size_t)n * 4));
    return from_cuda(sc::launch_slots_release(in_use, n_slots, slot_ids, n, (cudaStream_t)stream));
}

sc_status shortconv_pool_copy(sc_dtype dtype, int H, int K, void *pool, int n_slots,
                              const int32_t *src_slots, const int32_t *dst_slots, int n,
                              void *stream) {
    const sc_status st = check_shape(dtype, H, K);
    if (st != SC_OK) return st;
    if (n_slots <= 0 || n < 0) return SC_EINVAL;
    const int64_t state_bytes = (int64_t)H * K * elem_size(dtype);
    const size_t n_pool = (size_t)n_slots * state_bytes;
    if (!ptr_ok(pool, n_pool, 16) || !ptr_ok(src_slots, (size_t)n * 4, 4) ||
        !ptr_ok(dst_slots, (size_t)n * 4, 4))
        return SC_EINVAL;
    if (overlaps(pool, n_pool, src_slots, (size_t)n * 4) ||
        overlaps(pool, n_pool, dst_slots, (size_t)n * 4))
        return SC_EINVAL;
    if (n == 0) return SC_OK;
    SC_BOUNDS_INSTALL(kUnitSlots, RW(pool, n_pool), RO(src_slots, (size_t)n * 4),
                      RO(dst_slots, (size_t)n * 4));
    return from_cuda(sc::launch_pool_copy(src_slots, dst_slots, n, state_bytes, pool, n_slots,
                                          (cudaStream_t)stream));
}

sc_status shortconv_check_wait_limit(void *stream) {
    return from_cuda(sc::launch_wait_limit_check((cudaStream_t)stream));
}

sc_status shortconv_get_error(void *stream, int *device_code) {
    if (device_code == nullptr) return SC_EINVAL;
    unsigned int code = 0;
    const cudaError_t e = sc::read_and_clear_error((cudaStream_t)stream, &code);
    if (e != cudaSuccess) return SC_ECUDA;
    *device_code = (int)code;
    return code == 0 ? SC_OK : SC_EDEVICE;
}

int shortconv_bounds_checked(void) {
#ifdef SC_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

sc_status shortconv_bounds_trim_next(int region, uint64_t bytes) {
#ifdef SC_BOUNDS_CHECK
    if (region < 0 || region >= sc::kMaxBoundsRegions) return SC_EINVAL;
    std::lock_guard<std::mutex> lock(g_trim_mu);
    g_trim_index = region;
    g_trim_bytes = bytes;
    return SC_OK;
#else
    (void)region;
    (void)bytes;
    return SC_EUNSUPPORTED;
#endif
}

sc_status shortconv_bounds_take_first_bad(void *stream, uint64_t *addr) {
#ifdef SC_BOUNDS_CHECK
    if (addr == nullptr) return SC_EINVAL;
    unsigned long long a = 0;
    const cudaError_t e = sc::bounds_take_first_bad((cudaStream_t)stream, &a);
    if (e != cudaSuccess) return SC_ECUDA;
    *addr = (uint64_t)a;
    return SC_OK;
#else
    (void)stream;
    (void)addr;
    return SC_EUNSUPPORTED;
#endif
}

const char *shortconv_status_string(sc_status status) {
    switch (status) {
        case SC_OK: return "ok";
        case SC_EINVAL: return "invalid argument";
        case SC_EUNSUPPORTED: return "unsupported dtype or size";
        case SC_ECUDA: return "CUDA runtime error";
        case SC_EDEVICE: return "device-side data error (see the device error code)";
        default: return "unknown status";
    }
}

}  // extern "C"
