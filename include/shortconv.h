/*
 * shortconv.h -- C ABI of libshortconv.so: the LFM2 gated short convolution
 * ("ShortConv") hot path on GB300 (sm_103a).
 *
 * The operation (MAX Pipelines LFM2 article, "MAX Pipelines 的 LFM2 架构支持：
 * 混合全注意力 + 短卷积解码器实现解析", section "短卷积实现（LFM2ShortConv）"):
 * the in_proj output of a token is split into B, C and x; u = B * x; a
 * per-sequence window of the last K values of u slides by one per token
 * (oldest dropped, u appended); z = sum_k w[h,k] * window[k]; y = C * z.
 * Tap k = K-1 multiplies the newest value. There is no activation. The
 * per-channel conv bias is optional: NULL for the released LFM2
 * configurations, which are bias-free (Liger-Kernel PR #1317, "Kernel
 * changes / Gated short convolution"); when given, z = sum + b before the C
 * gate.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, contiguous):
 *   bcx   [T, 3H]         in_proj output, columns B | C | x
 *   w     [H, K]          depthwise conv weight
 *   pool  [n_slots, H, K] conv-state pool; slot s, channel h holds the last K
 *                         values of u (index K-1 newest). The pool stores u
 *                         after rounding to the pool dtype, exactly as the
 *                         convolution consumed it.
 *   y     [T, H]          output
 * dtype: bcx, w, pool, y (and win, dy, dbcx) all share one dtype, SC_F32 or
 *   SC_BF16. Products B*x are rounded once to that dtype to form u; the sum
 *   over taps and C*z are computed in fp32 and y is rounded once to the dtype.
 * Pointers: every array pointer is a DEVICE pointer (cudaMalloc'd or
 *   equivalent, e.g. a torch CUDA tensor's data pointer) on the current
 *   device, 16-byte aligned; int32 index arrays need 4-byte alignment. A
 *   pointer may be NULL only when the array it describes is empty.
 * Sizes: H > 0 and a multiple of 8; 1 <= K <= 4.
 * Ownership: the caller owns every buffer. The library allocates no device
 *   or host memory and keeps no pointer after a call returns.
 * Execution: every call only enqueues work on `stream` (a cudaStream_t; NULL
 *   means the legacy default stream) and returns without synchronizing,
 *   except shortconv_get_error.
 * Aliasing: no output may overlap any input of the same call, except the
 *   pool, which is read and written in place where stated.
 * Errors: argument errors are found on the host; the call then returns
 *   SC_EINVAL or SC_EUNSUPPORTED and enqueues nothing. A failed launch
 *   returns SC_ECUDA. Errors in DEVICE-resident data (slot ids, cu_seqlens,
 *   accepted lengths) cannot be seen by the host without a synchronization,
 *   so the kernels record them in a per-device error word (a bit mask of
 *   SC_DEV_* codes) and skip the offending unit; shortconv_get_error()
 *   returns and clears that word. No kernel traps or asserts.
 * Slot ids within one call must be distinct (not checked).
 */
#ifndef LFM2_SHORTCONV_H
#define LFM2_SHORTCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SC_OK = 0,
    SC_EINVAL = 1,        /* bad argument: null/misaligned pointer, bad size, overlap */
    SC_EUNSUPPORTED = 2,  /* valid request outside what is built (dtype, K, H % 8) */
    SC_ECUDA = 3,         /* a CUDA runtime call or launch failed */
    SC_EDEVICE = 4        /* shortconv_get_error found device-side errors */
} sc_status;

typedef enum { SC_F32 = 0, SC_BF16 = 1 } sc_dtype;

/* Bits of the device error word. */
#define SC_DEV_BAD_SLOT 0x1u      /* a slot id outside [0, n_slots): that sequence skipped */
#define SC_DEV_BAD_SEQLENS 0x2u   /* cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T: call skipped */
#define SC_DEV_BAD_ACCEPTED 0x4u  /* an accepted length outside [0, D]: that sequence skipped */
#define SC_DEV_TIMEOUT 0x8u       /* a bounded wait on an asynchronous copy gave up: output incomplete */
#define SC_DEV_NO_SLOT 0x10u      /* a claim asked for more slots than were free: nothing claimed */
#define SC_DEV_OUT_OF_BOUNDS 0x20u /* bounds-checked build only: an access outside the call's
                                      buffers was refused (see shortconv_bounds_checked) */

/*
 * The optional conv bias. Every forward and backward call below takes
 * `bias`: device [H] of the call's dtype, 16-byte aligned, read only; NULL
 * means no bias. A bias is added to the depthwise conv output of its channel
 * before the C gate: z_t = sum_k w_k u_{t-K+1+k} + bias[h], y_t = C_t z_t
 * (the MAX LFM2 article, section "批处理与权重适配", maps a checkpoint's
 * conv.conv.bias to the layer's conv_bias; the SGLang PR #31041 verify code,
 * section "实现拆解 2", passes conv_bias to the conv update with no
 * activation and gates by C afterwards). The released LFM2 checkpoints have
 * no conv bias; NULL gives exactly the bias-free results. With a bias, the
 * sum is rounded once in fp32 after the K-tap chain.
 */

/*
 * Packed variable-length prefill (continued prefill from each slot's state).
 *
 * Sequence i (0 <= i < N) is rows cu_seqlens[i] .. cu_seqlens[i+1]-1 of bcx
 * and y. Its history before its first row is the state in pool slot
 * slot_ids[i]; after the call that slot holds the last K values of u of the
 * sequence appended to its old state (for a sequence shorter than K the old
 * values that remain are kept). No history crosses a sequence boundary
 * ("feat(model): support LFM2-1.2B", section "供审阅者关注的事项"). A fresh
 * sequence is given a zeroed slot by the caller. Empty sequences leave their
 * slot unchanged. Slots not named in slot_ids are not touched.
 *
 *   dtype       SC_F32 or SC_BF16
 *   H, K        channels, taps
 *   bcx         device [T, 3H]           read
 *   T           total rows, 0 <= T < 2^31
 *   w           device [H, K]            read
 *   bias        device [H] or NULL       read (see above)
 *   cu_seqlens  device int32 [N + 1]     read; must be 0, non-decreasing, end at T
 *   N           number of sequences, >= 0 (N = 0 requires T = 0)
 *   slot_ids    device int32 [N]         read
 *   pool        device [n_slots, H, K]   read and written in place
 *   y           device [T, H]            written
 * Device errors: SC_DEV_BAD_SEQLENS (nothing is written), SC_DEV_BAD_SLOT
 * (that sequence's rows of y and its slot are not written), SC_DEV_TIMEOUT
 * (an asynchronous row copy did not complete within 2 s; output incomplete).
 *
 * Implementation: persistent CTAs (as many per SM as fit, 4 or 5 at bf16)
 * each stream a balanced range of rows of a 512-channel slice through
 * shared memory with bulk asynchronous copies (see shortconv_prefill_tiled
 * for the register-tiled alternative; both give identical bits).
 */
sc_status shortconv_prefill(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                            const void *w, const void *bias, const int32_t *cu_seqlens, int N,
                            const int32_t *slot_ids, void *pool, int n_slots, void *y,
                            void *stream);

/*
 * shortconv_prefill computed by the register-tiled kernel: each thread loads
 * and computes 8 channels of `rows_per_thread` consecutive rows (one of 4, 8,
 * 16, 32) straight from global memory; 0 means shortconv_prefill's streamed
 * kernel. Every choice gives identical bits; only the speed differs.
 */
sc_status shortconv_prefill_tiled(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                  const void *w, const void *bias, const int32_t *cu_seqlens,
                                  int N, const int32_t *slot_ids, void *pool, int n_slots,
                                  void *y, int rows_per_thread, void *stream);

/*
 * Decode: one new token per sequence, in place on the pool.
 *
 * Row i of bcx is the next token of sequence i, whose state lives in slot
 * slot_ids[i]. The slot's window slides by one and y[i] is that token's
 * output: the MAX per-token loop ("短卷积实现（LFM2ShortConv）": gather the
 * request's state, drop the oldest column, append bx_t, scatter back) for a
 * single token.
 *
 *   bcx [N, 3H] read; w [H, K] read; bias [H] or NULL read;
 *   slot_ids int32 [N] read; pool [n_slots, H, K] read and written;
 *   y [N, H] written.
 * Device errors: SC_DEV_BAD_SLOT (that sequence skipped).
 */
sc_status shortconv_decode(sc_dtype dtype, int H, int K, const void *bcx, int N,
                           const void *w, const void *bias, const int32_t *slot_ids,
                           void *pool, int n_slots, void *y, void *stream);

/*
 * Speculative verify: D draft tokens per sequence, recording the conv window
 * after every draft step (SGLang PR #31041, section "实现拆解 2": the target
 * verify pass writes each step's conv window to a speculative tape so that
 * the state can be rolled back to the accepted boundary).
 *
 * Rows i*D .. i*D+D-1 of bcx are sequence i's drafts, taken in order from
 * the state in slot slot_ids[i]. After draft j the K-wide window (what the
 * slot would hold had the sequence accepted j+1 drafts) is written to
 * win[i, j, :, :] and the draft's output to y[i*D + j]. The pool is only
 * read; shortconv_rollback commits the accepted prefix.
 *
 *   bcx [N*D, 3H] read; w [H, K] read; bias [H] or NULL read;
 *   slot_ids int32 [N] read; pool [n_slots, H, K] read;
 *   win [N, D, H, K] written; y [N*D, H] written.
 * Device errors: SC_DEV_BAD_SLOT (that sequence's win and y rows not written).
 */
sc_status shortconv_verify(sc_dtype dtype, int H, int K, const void *bcx, int N, int D,
                           const void *w, const void *bias, const int32_t *slot_ids,
                           const void *pool, int n_slots, void *win, void *y, void *stream);

/*
 * Rollback after verify: sequence i accepted accepted[i] of its D drafts
 * (0 <= accepted[i] <= D). For accepted[i] >= 1, win[i, accepted[i]-1]
 * becomes the state of slot slot_ids[i]; for 0 the slot keeps the state it
 * had before verify (verify does not modify the pool).
 *
 *   win [N, D, H, K] read (from shortconv_verify); accepted int32 [N] read;
 *   slot_ids int32 [N] read; pool [n_slots, H, K] written.
 * Device errors: SC_DEV_BAD_ACCEPTED, SC_DEV_BAD_SLOT (that sequence skipped).
 */
sc_status shortconv_rollback(sc_dtype dtype, int H, int K, int N, int D, const void *win,
                             const int32_t *accepted, const int32_t *slot_ids, void *pool,
                             int n_slots, void *stream);

/*
 * shortconv_rollback for L layers in one launch. A sequence's accepted length
 * is the same in every layer (acceptance is decided per sequence from the
 * model's output), so a serving loop rolls back all layers' states at once
 * after verify instead of one launch per layer. Layer l's verify tape is
 * win + l * N*D*H*K elements and its pool pool + l * n_slots*H*K elements:
 * stacked tapes and pools, each layer laid out as shortconv_rollback's.
 *
 *   win [L, N, D, H, K] read; accepted int32 [N] read; slot_ids int32 [N]
 *   read; pool [L, n_slots, H, K] written. L >= 1; L = 1 is shortconv_rollback.
 * Device errors: as shortconv_rollback (flagged once, for all layers).
 */
sc_status shortconv_rollback_layers(sc_dtype dtype, int H, int K, int L, int N, int D,
                                   const void *win, const int32_t *accepted,
                                   const int32_t *slot_ids, void *pool, int n_slots,
                                   void *stream);

/*
 * Bytes of device workspace shortconv_backward and shortconv_backward_varlen
 * need for these sizes (fp32 partial weight and bias gradients, one block per
 * row range). Host-only; no CUDA call; depends only on the arguments.
 * Returns 0 for invalid sizes.
 */
size_t shortconv_backward_workspace_bytes(int H, int K, int64_t T);

/*
 * Backward of one sequence of T rows that started from a zero state (the
 * training path: Liger-Kernel PR #1317, "Kernel changes / Gated short
 * convolution": the B/C gate gradients fused with the depthwise-conv input
 * gradient, and the weight gradient of all K taps of a channel reduced
 * together). With z_t = sum_k w_k u_{t-K+1+k} (+ bias[h]; u before row 0 is 0):
 *   dC_t = dy_t z_t;  dz_t = dy_t C_t;  du_s = sum_k w_k dz_{s+K-1-k}
 *   (terms past row T-1 are 0);  dB_s = du_s x_s;  dx_s = du_s B_s;
 *   dW[h,k] = sum_t dz_t u_{t-K+1+k};  dbias[h] = sum_t dz_t.
 * The rounding of u is passed straight through.
 *
 *   bcx [T, 3H] read; w [H, K] read; bias [H] or NULL read; dy [T, H] read;
 *   dbcx [T, 3H] written (dB | dC | dx, same dtype as bcx);
 *   dw [H, K] fp32 written (overwritten, not accumulated);
 *   dbias [H] fp32 written, or NULL (not computed; independent of bias);
 *   workspace: device scratch of at least
 *   shortconv_backward_workspace_bytes(H, K, T) bytes, 16-byte aligned,
 *   owned by the caller, contents ignored on entry and unspecified after.
 * The weight and bias gradients are reduced in a fixed order: repeated calls
 * give identical bits.
 */
sc_status shortconv_backward(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                             const void *w, const void *bias, const void *dy, void *dbcx,
                             float *dw, float *dbias, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Backward of the packed varlen prefill with initial states: training on
 * packed sequences, and chunked training that carries each sequence's state
 * from one chunk to the next (Liger-Kernel PR #1317's packed SFT workloads
 * train this layer on packed sequences; the zero-state single-sequence case
 * is shortconv_backward).
 *
 * Sequence i is rows cu_seqlens[i] .. cu_seqlens[i+1]-1 and starts from the
 * state init_states[i] (as a prefill would have read it from its slot). With
 * ext = [init_0 .. init_{K-1}, u_0 .. u_{len-1}], row t's window is
 * ext[t+1 .. t+K] and the final state is ext[len .. len+K-1]. Given dy and an
 * optional gradient d_final of the final states, the call writes
 *   dB, dC, dx (as shortconv_backward, history and look-ahead staying inside
 *   each sequence), dW and dbias (fp32, summed over all sequences) and
 *   d_init[i][h][m] = gradient of init_states[i][h][m] (tap 0 only ever gets
 *   d_final's share, for empty sequences).
 * The rounding of u is passed straight through.
 *
 *   bcx [T, 3H], w [H, K], dy [T, H]: read (dtype)
 *   bias [H] (dtype) or NULL: read
 *   cu_seqlens int32 [N + 1]: read; 0, non-decreasing, ending at T
 *   init_states [N, H, K] (dtype) or NULL for zero states: read
 *   d_final [N, H, K] fp32 or NULL for zero: read
 *   dbcx [T, 3H] (dtype), dw [H, K] fp32: written
 *   dbias [H] fp32 or NULL (not computed): written
 *   d_init [N, H, K] fp32 or NULL (not computed): written
 *   workspace: at least shortconv_backward_workspace_bytes(H, K, T) bytes.
 * Device errors: SC_DEV_BAD_SEQLENS (dw and dbias are zeroed; dbcx and
 * d_init are not written).
 */
sc_status shortconv_backward_varlen(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                    const void *w, const void *bias, const int32_t *cu_seqlens,
                                    int N, const void *init_states, const void *dy,
                                    const float *d_final, void *dbcx, float *dw, float *dbias,
                                    float *d_init, void *workspace, size_t workspace_bytes,
                                    void *stream);

/*
 * shortconv_backward without a workspace argument, for callers that cannot
 * allocate device memory when they call: code running inside a host
 * framework that owns all device memory through its own pool and forbids
 * direct cudaMalloc, and latency-critical paths where an allocation's
 * implicit device-wide synchronization, or an out-of-memory failure in the
 * middle of a step, is not acceptable. The pages have no counterpart to this
 * call; it only moves the scratch.
 *
 * Same results and bits as shortconv_backward with bias = dbias = NULL, and
 * its arguments less those and the workspace. The fp32 dW partials live in
 * a fixed 8 MiB device array inside the library, which every GPU that loads
 * the library holds until the process exits. The call allocates nothing and
 * never calls cudaMalloc or cudaFree.
 *   - Sizes whose dW partials exceed 8 MiB are rejected with
 *     SC_EUNSUPPORTED before anything is enqueued. The partials take
 *     min(ceil(T / 16), 152) * H * K * 4 bytes, so nothing is rejected
 *     for H * K <= 13,797 (every T for H = 2048 or H = 4096 with K = 3);
 *     for H = 8192, K = 4 rows above T = 1024 are.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for
 *     the life of the process; make that first call before any stream
 *     capture on that device. A device reset (cudaDeviceReset) or a context
 *     torn down and created again after that first call is not supported:
 *     the cached address would no longer be the array's.
 *   - All calls on a device share the one array and each overwrites it
 *     before reading it, so no clearing is needed; calls that overlap on the
 *     GPU (for instance on two streams) race on it and must be serialized
 *     by the caller.
 */
sc_status shortconv_backward_noalloc(sc_dtype dtype, int H, int K, const void *bcx, int64_t T,
                                     const void *w, const void *dy, void *dbcx, float *dw,
                                     void *stream);

/*
 * The layer's projections on the tensor cores (bf16 only).
 *
 * The MAX LFM2 article (section "短卷积实现（LFM2ShortConv）") gives the
 * layer: in_proj maps the hidden state to three parts b, c, xv; bx = b * xv
 * goes through the causal conv; y = c * conv_out goes through out_proj.
 * Neither projection has a bias there. A projection from n to m features
 * has the weight [m, n] (row-major), so in_proj's is [3H, D] (rows 0..H-1
 * give b, H..2H-1 c, 2H..3H-1 xv) and out_proj's is [D, H].
 *
 * shortconv_in_proj_prefill computes in_proj and the whole packed varlen
 * prefill of shortconv_prefill in one pass: the [T, 3H] projection is
 * accumulated in fp32, rounded to bf16 (the values a separate in_proj
 * would store) and consumed in the GEMM's epilogue; it never reaches
 * memory. Results are those of shortconv_prefill on that projection, so
 * they differ from in_proj followed by shortconv_prefill only where the
 * fp32 accumulation order of the projection changes a bf16 rounding.
 *
 *   D, H, K      model width (D % 64 == 0), channels (H % 64 == 0), taps
 *   hidden       device [T, D] bf16            read
 *   w_in         device [3H, D] bf16           read
 *   w, bias      as shortconv_prefill (bias [H] or NULL)
 *   cu_seqlens, N, slot_ids, pool, n_slots, y: as shortconv_prefill
 *   workspace    device scratch of at least
 *                shortconv_in_proj_workspace_bytes(H, K, N) bytes, 16-byte
 *                aligned, owned by the caller (the last K values of u per
 *                sequence, from which a second pass writes the slots' new
 *                states after all rows are done; a call with one sequence
 *                usually writes its state in the fused pass and leaves the
 *                workspace untouched)
 * Device errors: as shortconv_prefill, plus SC_DEV_TIMEOUT (a bounded wait
 * on a tensor copy or on the tensor cores gave up; output incomplete).
 */
size_t shortconv_in_proj_workspace_bytes(int H, int K, int N);
sc_status shortconv_in_proj_prefill(sc_dtype dtype, int D, int H, int K, const void *hidden,
                                    int64_t T, const void *w_in, const void *w, const void *bias,
                                    const int32_t *cu_seqlens, int N, const int32_t *slot_ids,
                                    void *pool, int n_slots, void *y, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * shortconv_in_proj_decode: in_proj fused with shortconv_decode, for the
 * serving decode step (one token per sequence). The MAX LFM2 article
 * (section "短卷积实现（LFM2ShortConv）") gives the per-token step: gather
 * the sequence's conv state, slide in bx = b * xv, take the weighted sum,
 * gate by c, scatter the state back. Here row i of `hidden` is the one
 * token of sequence i: its [B | C | x] projection is accumulated in fp32 on
 * the tensor cores, rounded to bf16 and consumed in the GEMM's epilogue
 * (never stored), and the conv state of slot slot_ids[i] is read and written
 * in the same pass. One launch, no workspace. Results are those of
 * shortconv_decode on that bf16 projection.
 *
 *   D, H, K      model width (D % 64 == 0), channels (H % 64 == 0), taps
 *   hidden       device [N, D] bf16            read
 *   N            sequences (rows), >= 0
 *   w_in         device [3H, D] bf16           read (rows b | c | xv)
 *   w, bias      device [H, K] bf16; bias [H] bf16 or NULL
 *   slot_ids     device int32 [N]              read; distinct
 *   pool         device [n_slots, H, K] bf16   read and written in place
 *   y            device [N, H] bf16            written
 * Device errors: SC_DEV_BAD_SLOT (that sequence's y row and slot are not
 * written), SC_DEV_TIMEOUT (a bounded wait on a tensor copy or on the tensor
 * cores gave up; output incomplete).
 */
sc_status shortconv_in_proj_decode(sc_dtype dtype, int D, int H, int K, const void *hidden,
                                   int N, const void *w_in, const void *w, const void *bias,
                                   const int32_t *slot_ids, void *pool, int n_slots, void *y,
                                   void *stream);

/*
 * out_proj: out = y w_out^T, fp32 accumulation, rounded once to bf16.
 *   y [T, H] bf16 read (H % 64 == 0); w_out [D, H] bf16 read
 *   (D % 256 == 0); out [T, D] bf16 written.
 */
sc_status shortconv_out_proj(sc_dtype dtype, int H, int D, const void *y, int64_t T,
                             const void *w_out, void *out, void *stream);

/*
 * Conv-state slot pool on the device (MAX LFM2 article, section "推理状态管理：
 * ConvStateCache 与卷积状态生命周期": a request claims a free slot -- an error
 * when none is free --, starts from a zero state, and releases the slot when
 * it finishes). The in-use set is a caller-owned device bitmap of
 * (n_slots + 31) / 32 uint32 words, bit (s % 32) of word s / 32 set while slot
 * s is in use; bits past n_slots are ignored and kept. Calls on one bitmap
 * must be ordered (one stream), like any read-modify-write of device memory.
 *
 * shortconv_slots_claim: take the n_claim lowest-numbered free slots, in
 * increasing order, mark them in use and write them to slots_out [n_claim];
 * if pool is not NULL (a [n_slots, H, K] pool of `dtype`) their states are
 * zeroed. All-or-nothing: with fewer than n_claim free slots nothing is
 * claimed, slots_out is all -1 and SC_DEV_NO_SLOT is set. 0 <= n_claim <= n_slots.
 */
sc_status shortconv_slots_claim(uint32_t *in_use, int n_slots, int n_claim, int32_t *slots_out,
                                sc_dtype dtype, int H, int K, void *pool, void *stream);

/*
 * shortconv_slots_release: mark slot_ids [n] free. An id out of range or not
 * in use sets SC_DEV_BAD_SLOT and is skipped; the others are released.
 */
sc_status shortconv_slots_release(uint32_t *in_use, int n_slots, const int32_t *slot_ids, int n,
                                  void *stream);

/*
 * shortconv_pool_copy: pool[dst_slots[i]] = pool[src_slots[i]] for i < n (a
 * state snapshot, e.g. to reuse the state reached at a shared prefix).
 * Destinations must be distinct and not among the sources (not checked). An
 * id out of range sets SC_DEV_BAD_SLOT and skips that pair.
 */
sc_status shortconv_pool_copy(sc_dtype dtype, int H, int K, void *pool, int n_slots,
                              const int32_t *src_slots, const int32_t *dst_slots, int n,
                              void *stream);

/*
 * shortconv_check_wait_limit: a health check of the device-side timeout path,
 * which a working call never reaches. Every waiting kernel of this library
 * bounds each wait on an asynchronous copy or on the tensor cores (about 2 s),
 * then sets SC_DEV_TIMEOUT and returns instead of hanging. This call enqueues
 * a one-thread kernel that waits, with that same bounded wait, on a device
 * barrier that nothing ever completes: about 2 s later it sets SC_DEV_TIMEOUT
 * and returns, and shortconv_get_error reports it. The device stays usable.
 * Not part of the pages' interface. Errors: SC_ECUDA if the launch fails.
 */
sc_status shortconv_check_wait_limit(void *stream);

/*
 * Synchronize `stream`, then read and clear the current device's error word.
 * *device_code receives the SC_DEV_* bits seen since the last clear (0 if
 * none). Returns SC_OK if the word was 0, SC_EDEVICE if not, SC_ECUDA if a
 * CUDA call failed, SC_EINVAL if device_code is NULL. The word is shared by
 * all streams on the device.
 */
sc_status shortconv_get_error(void *stream, int *device_code);

/* Static, never-NULL description of a status code. */
const char *shortconv_status_string(sc_status status);

/*
 * The bounds-checked build. The library can also be built with
 * -DSC_BOUNDS_CHECK (python -m lfm2_gated_short_gb300.build --bounds-check,
 * into _build/bounds/). In that build every entry point first records the
 * buffers the call may read and write (its arguments, with the sizes the
 * call implies), and every global load and store the kernels make through
 * their memory helpers checks that its whole byte range lies in one of them
 * (stores: in a writable one). A refused access is skipped -- a load reads
 * zeros, a store writes nothing, a bulk copy is not issued -- and sets
 * SC_DEV_OUT_OF_BOUNDS in the error word; nothing traps. Tiled tensor copies
 * (the projections' operand loads) are bounded by their tensor maps instead.
 * The records are per library instance, so calls that overlap on the GPU
 * must not be made in this build. It is slower and meant for tests; the
 * pages have no counterpart to it.
 *
 * shortconv_bounds_checked: 1 in the bounds-checked build, 0 otherwise.
 *
 * shortconv_bounds_trim_next: shorten, by `bytes`, buffer number `region`
 * of the next call's record (buffers are numbered in the order each entry
 * point lists them: for shortconv_prefill bcx 0, w 1, bias 2, cu_seqlens 3,
 * slot_ids 4, pool 5, y 6), so that its last bytes count as outside the
 * call. This shows the checks at work without any real out-of-bounds
 * access: the memory is still there, only the record is shorter.
 * SC_EINVAL for a region number outside [0, 16); SC_EUNSUPPORTED in the
 * standard build.
 *
 * shortconv_bounds_take_first_bad: synchronize `stream` and return in
 * *addr the first device address refused since the last take (0 if none),
 * clearing it. SC_EUNSUPPORTED in the standard build.
 */
int shortconv_bounds_checked(void);
sc_status shortconv_bounds_trim_next(int region, uint64_t bytes);
sc_status shortconv_bounds_take_first_bad(void *stream, uint64_t *addr);

#ifdef __cplusplus
}
#endif

#endif /* LFM2_SHORTCONV_H */
