/*
 * shortconv_oracle.c -- plain, slow, scalar CPU oracle for the LFM2 gated
 * short convolution (ShortConv).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. The product
 * path never calls it and shares no code, header or constant with it.
 *
 * What it computes follows the operational definition on
 *   "MAX Pipelines 的 LFM2 架构支持：混合全注意力 + 短卷积解码器实现解析",
 *   section "短卷积实现（LFM2ShortConv）":
 *     in_proj splits into b, c, xv; bx = b * xv; for every token the
 *     request's [1, hidden, K] state drops its oldest column and appends
 *     bx_t (concat(state[:, :, 1:], bx_t)); conv_out = sum(state * w, K);
 *     y = c * conv_out.
 * and the state rules of the same page's section "推理状态管理：ConvStateCache
 * 与卷积状态生命周期" (one [hidden, K] state per request slot).
 *
 * Speculative verify / rollback follows "SGLang PR #31041" (LFM2 DSpark),
 * section "实现拆解 2 (LFM2 目标侧 TARGET_VERIFY：ShortConv 验证与回滚)":
 * the conv window after every draft step is recorded, and after verification
 * the state is restored at the accepted boundary.
 *
 * The backward pass follows "[Feature] Add LFM2, LFM2-MoE, and LFM2-VL
 * support" (Liger-Kernel PR #1317), section "Kernel changes / Gated short
 * convolution": gradients of the B/C gates and the depthwise conv input, and
 * a per-channel weight gradient holding all K taps, bias-free.
 *
 * Every value is carried in double. The only roundings are the ones the
 * stored data types force:
 *   u = round(B * x)      -- the value that enters the state (stored dtype)
 *   y = round(C * z)      -- one rounding of the output, z kept in double
 * dtype ORC_F64 is a test-only mode in which round() is the identity.
 *
 * bf16 <-> double conversions are written out below from the IEEE-754
 * binary32 layout (bf16 = the upper 16 bits of a binary32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_EDATA = 4 };

/* ---------------------------------------------------------------- dtypes */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16 value, ties to even, in ONE rounding
 * step. bf16 keeps 8 significant bits and binary32's exponent range, so the
 * spacing of bf16 values around |d| in [2^e, 2^(e+1)) is 2^(e-7), and below
 * the smallest normal (2^-126) it stays 2^-133.
 */
uint16_t orc_double_to_bf16(double d)
{
    if (isnan(d))
        return 0x7FC0;
    if (isinf(d))
        return signbit(d) ? 0xFF80 : 0x7F80;
    if (d == 0.0)
        return signbit(d) ? 0x8000 : 0x0000;
    int e = ilogb(d);
    if (e < -126)
        e = -126;
    double spacing = ldexp(1.0, e - 7);
    double r = nearbyint(d / spacing) * spacing; /* default mode: ties to even */
    const double bf16_max = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max)
        return signbit(d) ? 0xFF80 : 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

double orc_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

/* orc_double_to_bf16 over an array of n values. */
void orc_round_bf16_array(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_double_to_bf16(in[i]);
}

static double round_to(int dt, double v)
{
    switch (dt) {
    case ORC_F32:
        return (double)(float)v;
    case ORC_BF16:
        return bf16_bits_to_double(orc_double_to_bf16(v));
    default:
        return v;
    }
}

static double load(int dt, const void *p, int64_t i)
{
    switch (dt) {
    case ORC_F32:
        return (double)((const float *)p)[i];
    case ORC_BF16:
        return bf16_bits_to_double(((const uint16_t *)p)[i]);
    default:
        return ((const double *)p)[i];
    }
}

static void store(int dt, void *p, int64_t i, double v)
{
    switch (dt) {
    case ORC_F32:
        ((float *)p)[i] = (float)v;
        break;
    case ORC_BF16:
        ((uint16_t *)p)[i] = orc_double_to_bf16(v);
        break;
    default:
        ((double *)p)[i] = v;
        break;
    }
}

static int dtype_ok(int dt) { return dt == ORC_F32 || dt == ORC_BF16 || dt == ORC_F64; }

/* ----------------------------------------------------------- forward core */

/*
 * One sequence, one channel h: the per-token sliding window of the MAX
 * definition. An optional per-channel bias (NULL: none) is added to the conv
 * output before the C gate, the place conv1d's bias takes in the SGLang verify
 * listing (causal_conv1d_update(..., conv_bias, activation=None), gated by C
 * afterwards). win[0..K-1] enters holding the slot's state (oldest first) and
 * leaves holding the last K values of [state; u_0 .. u_{len-1}].
 * Row t of bcx is [B(0..H-1) | C(H..2H-1) | x(2H..3H-1)].
 */
static void run_channel(int dt, int H, int K, const void *bcx, int64_t row0,
                        int64_t len, const void *w, const void *bias, int h, double *win,
                        void *y, int64_t y_row0)
{
    for (int64_t r = 0; r < len; ++r) {
        int64_t t = row0 + r;
        double b = load(dt, bcx, t * 3 * H + h);
        double c = load(dt, bcx, t * 3 * H + H + h);
        double x = load(dt, bcx, t * 3 * H + 2 * H + h);
        double u = round_to(dt, b * x);
        for (int k = 0; k + 1 < K; ++k)
            win[k] = win[k + 1];
        win[K - 1] = u;
        double z = 0.0;
        for (int k = 0; k < K; ++k)
            z += load(dt, w, (int64_t)h * K + k) * win[k];
        if (bias)
            z += load(dt, bias, h);
        store(dt, y, (y_row0 + r) * H + h, c * z);
    }
}

/*
 * Packed varlen prefill. Sequence i covers rows cu_seqlens[i] .. cu_seqlens[i+1]-1
 * and owns pool slot slot_ids[i]; it reads that slot's state as its history
 * and writes its final state back. No history crosses a sequence boundary
 * ("feat(model): support LFM2-1.2B", section "供审阅者关注的事项": packed
 * prefill must not share ShortConv history between requests).
 *
 * Returns ORC_EDATA (and touches nothing) when cu_seqlens is not a
 * non-decreasing list from 0 to T. A sequence whose slot id is out of range
 * is skipped (its y rows and every slot stay untouched) and ORC_EDATA is
 * returned after the others are done.
 */
int orc_prefill(int dt, int H, int K, const void *bcx, int64_t T, const void *w,
                const void *bias, const int32_t *cu_seqlens, int N, const int32_t *slot_ids,
                void *pool, int n_slots, void *y)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || T < 0 || N < 0 || n_slots <= 0)
        return ORC_EINVAL;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T)
        return ORC_EDATA;
    for (int i = 0; i < N; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i])
            return ORC_EDATA;
    double *win = (double *)malloc(sizeof(double) * (size_t)K);
    if (!win)
        return ORC_EINVAL;
    int status = ORC_OK;
    for (int i = 0; i < N; ++i) {
        int s = slot_ids[i];
        if (s < 0 || s >= n_slots) {
            status = ORC_EDATA;
            continue;
        }
        int64_t row0 = cu_seqlens[i], len = (int64_t)cu_seqlens[i + 1] - cu_seqlens[i];
        for (int h = 0; h < H; ++h) {
            int64_t base = ((int64_t)s * H + h) * K;
            for (int k = 0; k < K; ++k)
                win[k] = load(dt, pool, base + k);
            run_channel(dt, H, K, bcx, row0, len, w, bias, h, win, y, row0);
            for (int k = 0; k < K; ++k)
                store(dt, pool, base + k, win[k]);
        }
    }
    free(win);
    return status;
}

/*
 * Decode: one new token per sequence, rows 0..N-1 of bcx, in place on the
 * pool. This is the prefill loop with one-token sequences.
 */
int orc_decode(int dt, int H, int K, const void *bcx, int N, const void *w, const void *bias,
               const int32_t *slot_ids, void *pool, int n_slots, void *y)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || N < 0 || n_slots <= 0)
        return ORC_EINVAL;
    double *win = (double *)malloc(sizeof(double) * (size_t)K);
    if (!win)
        return ORC_EINVAL;
    int status = ORC_OK;
    for (int i = 0; i < N; ++i) {
        int s = slot_ids[i];
        if (s < 0 || s >= n_slots) {
            status = ORC_EDATA;
            continue;
        }
        for (int h = 0; h < H; ++h) {
            int64_t base = ((int64_t)s * H + h) * K;
            for (int k = 0; k < K; ++k)
                win[k] = load(dt, pool, base + k);
            run_channel(dt, H, K, bcx, i, 1, w, bias, h, win, y, i);
            for (int k = 0; k < K; ++k)
                store(dt, pool, base + k, win[k]);
        }
    }
    free(win);
    return status;
}

/*
 * Speculative verify: sequence i owns draft rows i*D .. i*D+D-1. Starting
 * from its slot's state it takes the D steps in order; after step j the
 * K-wide window is recorded in win_out[i, j, :, :] (layout [N, D, H, K]) and
 * y gets the step's output. The pool is only read.
 */
int orc_verify(int dt, int H, int K, const void *bcx, int N, int D, const void *w,
               const void *bias, const int32_t *slot_ids, const void *pool, int n_slots,
               void *win_out, void *y)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || N < 0 || D <= 0 || n_slots <= 0)
        return ORC_EINVAL;
    double *win = (double *)malloc(sizeof(double) * (size_t)K);
    if (!win)
        return ORC_EINVAL;
    int status = ORC_OK;
    for (int i = 0; i < N; ++i) {
        int s = slot_ids[i];
        if (s < 0 || s >= n_slots) {
            status = ORC_EDATA;
            continue;
        }
        for (int h = 0; h < H; ++h) {
            int64_t base = ((int64_t)s * H + h) * K;
            for (int k = 0; k < K; ++k)
                win[k] = load(dt, pool, base + k);
            for (int j = 0; j < D; ++j) {
                int64_t t = (int64_t)i * D + j;
                run_channel(dt, H, K, bcx, t, 1, w, bias, h, win, y, t);
                for (int k = 0; k < K; ++k)
                    store(dt, win_out, (t * H + h) * K + k, win[k]);
            }
        }
    }
    free(win);
    return status;
}

/*
 * Rollback after verify: sequence i accepted a_i of its D drafts. For
 * a_i >= 1 the window recorded after draft a_i - 1 becomes the slot's state;
 * a_i = 0 leaves the slot as it was before verify. An out-of-range a_i or
 * slot id skips that sequence and returns ORC_EDATA.
 */
int orc_rollback(int dt, int H, int K, int N, int D, const void *win_in,
                 const int32_t *accepted, const int32_t *slot_ids, void *pool,
                 int n_slots)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || N < 0 || D <= 0 || n_slots <= 0)
        return ORC_EINVAL;
    int status = ORC_OK;
    for (int i = 0; i < N; ++i) {
        int a = accepted[i], s = slot_ids[i];
        if (a < 0 || a > D || s < 0 || s >= n_slots) {
            status = ORC_EDATA;
            continue;
        }
        if (a == 0)
            continue;
        int64_t src = (((int64_t)i * D + (a - 1)) * H) * K;
        int64_t dst = (int64_t)s * H * K;
        for (int64_t e = 0; e < (int64_t)H * K; ++e)
            store(dt, pool, dst + e, load(dt, win_in, src + e));
    }
    return status;
}

/* --------------------------------------------------------------- backward */

/*
 * Backward of y = C * conv(u), u = round(B * x), for one sequence of T rows
 * starting from a zero state (so the state carries no gradient), given the
 * upstream gradient dy [T, H]. With z_t = sum_k w_k u_{t-K+1+k} (u_{<0} = 0):
 *   dC_t   = dy_t * z_t
 *   dz_t   = dy_t * C_t
 *   du_s   = sum_k w_k dz_{s+K-1-k}        (terms past the last row are 0)
 *   dB_s   = du_s * x_s,   dx_s = du_s * B_s
 *   dW_h,k = sum_t dz_t u_{t-K+1+k}         (all K taps of a channel together)
 * The rounding of u is passed straight through (its derivative taken as 1).
 * dbcx has bcx's [T, 3H] layout (dB | dC | dx); dw is [H, K] in double. With
 * a bias (NULL: none) z_t includes it, and dbias[h] = sum_t dz_t (dbias NULL:
 * not written).
 */
int orc_backward(int dt, int H, int K, const void *bcx, int64_t T, const void *w,
                 const void *bias, const void *dy, void *dbcx, double *dw, double *dbias)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || T < 0)
        return ORC_EINVAL;
    size_t n = (size_t)(T > 0 ? T : 1);
    double *u = (double *)malloc(sizeof(double) * n);
    double *z = (double *)malloc(sizeof(double) * n);
    double *dz = (double *)malloc(sizeof(double) * n);
    if (!u || !z || !dz) {
        free(u);
        free(z);
        free(dz);
        return ORC_EINVAL;
    }
    for (int h = 0; h < H; ++h) {
        for (int64_t t = 0; t < T; ++t)
            u[t] = round_to(dt, load(dt, bcx, t * 3 * H + h) *
                                    load(dt, bcx, t * 3 * H + 2 * H + h));
        for (int64_t t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                int64_t p = t - K + 1 + k;
                if (p >= 0)
                    acc += load(dt, w, (int64_t)h * K + k) * u[p];
            }
            z[t] = bias ? acc + load(dt, bias, h) : acc;
        }
        for (int64_t t = 0; t < T; ++t) {
            double g = load(dt, dy, t * H + h);
            double c = load(dt, bcx, t * 3 * H + H + h);
            dz[t] = g * c;
            store(dt, dbcx, t * 3 * H + H + h, g * z[t]);
        }
        for (int64_t s = 0; s < T; ++s) {
            double du = 0.0;
            for (int k = 0; k < K; ++k) {
                int64_t q = s + K - 1 - k;
                if (q < T)
                    du += load(dt, w, (int64_t)h * K + k) * dz[q];
            }
            double b = load(dt, bcx, s * 3 * H + h);
            double x = load(dt, bcx, s * 3 * H + 2 * H + h);
            store(dt, dbcx, s * 3 * H + h, du * x);
            store(dt, dbcx, s * 3 * H + 2 * H + h, du * b);
        }
        for (int k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                int64_t p = t - K + 1 + k;
                if (p >= 0)
                    acc += dz[t] * u[p];
            }
            dw[(int64_t)h * K + k] = acc;
        }
        if (dbias) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t)
                acc += dz[t];
            dbias[h] = acc;
        }
    }
    free(u);
    free(z);
    free(dz);
    return ORC_OK;
}

/*
 * Backward of the packed varlen prefill with initial states (training on
 * packed sequences, and chunked training that carries the state from one
 * chunk to the next). Sequence i covers rows cu_seqlens[i] .. cu_seqlens[i+1]-1
 * and starts from the state init[i] ([N, H, K], NULL = zeros). Writing the
 * sequence as one array ext = [init_0 .. init_{K-1}, u_0 .. u_{len-1}], the
 * window at row t is ext[t+1 .. t+K], z_t = sum_k w_k ext[t+1+k] and the final
 * state is ext[len .. len+K-1]. Given dy and an optional gradient d_final
 * ([N, H, K] doubles, NULL = zeros) of the final states:
 *   d ext[j] = sum over (t, k) with t+1+k = j of w_k dz_t,  dz_t = dy_t C_t,
 *              plus d_final[j - len] for j >= len;
 *   du_s = d ext[K+s];  dB_s = du_s x_s;  dx_s = du_s B_s;  dC_t = dy_t z_t;
 *   dW[h,k] = sum over sequences and rows of dz_t ext[t+1+k];
 *   d_init[i] = d ext[0 .. K-1]  ([N, H, K] doubles, written if not NULL);
 * with a bias (NULL: none) z_t includes it and dbias[h] = sum of dz_t.
 * The rounding of u is passed straight through. Returns ORC_EDATA (nothing
 * written) for a cu_seqlens that is not 0 <= ... <= T ending at T.
 */
int orc_backward_varlen(int dt, int H, int K, const void *bcx, int64_t T, const void *w,
                        const void *bias, const int32_t *cu_seqlens, int N, const void *init,
                        const void *dy, const double *d_final, void *dbcx, double *dw,
                        double *dbias, double *d_init)
{
    if (!dtype_ok(dt) || H <= 0 || K <= 0 || T < 0 || N < 0)
        return ORC_EINVAL;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T)
        return ORC_EDATA;
    int64_t maxlen = 0;
    for (int i = 0; i < N; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i])
            return ORC_EDATA;
        if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen)
            maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
    }
    size_t n = (size_t)(K + maxlen);
    double *ext = (double *)malloc(sizeof(double) * n);
    double *dext = (double *)malloc(sizeof(double) * n);
    if (!ext || !dext) {
        free(ext);
        free(dext);
        return ORC_EINVAL;
    }
    for (int64_t e = 0; e < (int64_t)H * K; ++e)
        dw[e] = 0.0;
    if (dbias)
        for (int h = 0; h < H; ++h)
            dbias[h] = 0.0;
    for (int i = 0; i < N; ++i) {
        int64_t row0 = cu_seqlens[i], len = (int64_t)cu_seqlens[i + 1] - cu_seqlens[i];
        for (int h = 0; h < H; ++h) {
            int64_t sbase = ((int64_t)i * H + h) * K;
            for (int m = 0; m < K; ++m)
                ext[m] = init ? load(dt, init, sbase + m) : 0.0;
            for (int64_t s = 0; s < len; ++s) {
                int64_t r = row0 + s;
                ext[K + s] = round_to(dt, load(dt, bcx, r * 3 * H + h) *
                                              load(dt, bcx, r * 3 * H + 2 * H + h));
            }
            for (int64_t j = 0; j < K + len; ++j)
                dext[j] = 0.0;
            for (int64_t t = 0; t < len; ++t) {
                int64_t r = row0 + t;
                double z = 0.0;
                for (int k = 0; k < K; ++k)
                    z += load(dt, w, (int64_t)h * K + k) * ext[t + 1 + k];
                if (bias)
                    z += load(dt, bias, h);
                double g = load(dt, dy, r * H + h);
                double dz = g * load(dt, bcx, r * 3 * H + H + h);
                if (dbias)
                    dbias[h] += dz;
                store(dt, dbcx, r * 3 * H + H + h, g * z);
                for (int k = 0; k < K; ++k) {
                    dext[t + 1 + k] += load(dt, w, (int64_t)h * K + k) * dz;
                    dw[(int64_t)h * K + k] += dz * ext[t + 1 + k];
                }
            }
            if (d_final)
                for (int k = 0; k < K; ++k)
                    dext[len + k] += d_final[sbase + k];
            for (int64_t s = 0; s < len; ++s) {
                int64_t r = row0 + s;
                double du = dext[K + s];
                store(dt, dbcx, r * 3 * H + h, du * load(dt, bcx, r * 3 * H + 2 * H + h));
                store(dt, dbcx, r * 3 * H + 2 * H + h, du * load(dt, bcx, r * 3 * H + h));
            }
            if (d_init)
                for (int m = 0; m < K; ++m)
                    d_init[sbase + m] = dext[m];
        }
    }
    free(ext);
    free(dext);
    return ORC_OK;
}

