// proj.cu -- the ShortConv layer's projections on the tcgen05 tensor cores.
//
// The MAX LFM2 article (section "短卷积实现（LFM2ShortConv）") gives the layer:
// in_proj maps the hidden state to three parts b, c, xv; bx = b * xv goes
// through the causal depthwise conv; c * conv_out goes through out_proj.
//
// k_in_proj_conv fuses everything up to out_proj into the in_proj GEMM: a CTA
// computes the 128 x 192 product block [B | C | x] of 64 channels for 128
// rows (bf16 operands streamed by tiled TMA through a 4-stage ring, fp32
// accumulators in TMEM), and its epilogue rounds B, C, x to bf16 (the values
// a separate in_proj would store), forms u = round(B x), runs the K-tap conv
// over the tile's rows and writes y = round(C z). The [T, 3H] projection never
// reaches HBM. Consecutive row tiles overlap by K - 1 rows, so every output
// row finds its conv history in its own tile; at a sequence start the
// history comes from the sequence's slot.
//
// A tile holding a sequence's first rows reads the slot; another tile may
// hold its last rows. So the fused kernel writes the last K values of u of
// each sequence to a workspace, and k_commit_states (next in the stream)
// writes the new states: no tile writes a slot another tile reads.
//
// k_out_proj is the plain out_proj GEMM (128 x 256 tiles) on the same
// mainloop, with a store epilogue.
//
// Warp roles (192 threads): warp 0 issues the TMA copies, warp 1 owns the
// TMEM allocation and one of its lanes issues the MMAs, warps 2-5 run the
// epilogue (warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31). Every
// mbarrier wait gives up after 2 s (SC_DEV_TIMEOUT); the TMEM is always freed.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "errors.cuh"
#include "kernels.h"
#include "launch.h"
#include "shortconv.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace sc {

typedef __nv_bfloat16 bf16;

constexpr int kPBM = 128;                     // rows per tile = TMEM lanes
constexpr int kPBK = 64;                      // K per stage: one 128-byte swizzle row
constexpr int kPStages = 4;
constexpr int kPThreads = 192;
constexpr uint32_t kPTmemCols = 512;  // two 256-column accumulator buffers
constexpr uint32_t kPABytes = kPBM * kPBK * 2;  // 16 KB

constexpr int kConvCh = 64;                   // channels per fused tile
constexpr int kConvN = 3 * kConvCh;           // GEMM N: B | C | x of those channels
constexpr uint32_t kConvStage = kPABytes + kConvN * kPBK * 2;  // 40 KB
constexpr int kUStride = 144;                 // bytes per u row: 128 + 16, conflict-free
constexpr int kProjCuStaged = 512;

constexpr int kOutN = 256;                    // out_proj N per tile
constexpr uint32_t kOutStage = kPABytes + kOutN * kPBK * 2;    // 48 KB

// Shared memory after the stage ring: barriers and flags. The accumulator
// is double-buffered in TMEM (columns 0.. and 256..): the MMA lane fills one
// buffer while the epilogue warps drain the other.
struct PipeState {
    uint64_t full[kPStages];   // stage loaded (TMA bytes)
    uint64_t empty[kPStages];  // stage consumed (MMA commit)
    uint64_t tfull[2];         // accumulator buffer ready (MMA commit)
    uint64_t tempty[2];        // accumulator buffer drained (128 epilogue threads)
    uint64_t mma_done;         // every MMA of this CTA completed
    uint32_t tmem;
    volatile int abort;        // set by the producer or the MMA lane when a wait gave up
};

constexpr size_t kConvExtra = (size_t)kPBM * kUStride          // u tile
                              + kConvCh * 4 * sizeof(float)    // taps
                              + kConvCh * sizeof(float)        // bias
                              + (kProjCuStaged + 8) * 4;       // staged cu_seqlens
constexpr size_t conv_smem_bytes() {
    return 1024 + (size_t)kPStages * kConvStage + kConvExtra + sizeof(PipeState);
}
constexpr size_t out_smem_bytes() {
    return 1024 + (size_t)kPStages * kOutStage + sizeof(PipeState);
}

// ------------------------------------------------------------ persistent mainloop
//
// A CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ...; the stage ring
// runs on across tiles (k-block counter g over all of the CTA's tiles).

__device__ __forceinline__ void pipe_init(PipeState *ps) {
#pragma unroll
    for (int s = 0; s < kPStages; ++s) {
        mbar_init(&ps->full[s], 1);
        mbar_init(&ps->empty[s], 1);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        mbar_init(&ps->tfull[b], 1);
        mbar_init(&ps->tempty[b], 128);
    }
    mbar_init(&ps->mma_done, 1);
    ps->abort = 0;
    mbar_fence_init();
}

// Warp 0, one lane. coords(tile, a_row, b_rows) gives a tile's A row and the
// first rows of its NB boxes of B.
template <int NB, typename Coords>
__device__ __forceinline__ void produce_tiles(const CUtensorMap *ma, const CUtensorMap *mb,
                                              uint32_t stages, uint32_t stage_bytes,
                                              PipeState *ps, int nk, int n_tiles,
                                              uint32_t box_bytes, Coords coords) {
    uint32_t g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        int a_row, b_rows[NB];
        coords(tile, a_row, b_rows);
        for (int kb = 0; kb < nk; ++kb, ++g) {
            const uint32_t s = g % kPStages;
            if (g >= kPStages &&
                !mbar_wait_bounded(&ps->empty[s], (g / kPStages - 1) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                ps->abort = 1;
                ok = false;
                break;
            }
            const uint32_t st = stages + s * stage_bytes;
            mbar_arrive_expect_tx(&ps->full[s], kPABytes + NB * box_bytes);
            tma_load_2d(st, ma, &ps->full[s], kb * kPBK, a_row);
#pragma unroll
            for (int i = 0; i < NB; ++i)
                tma_load_2d(st + kPABytes + i * box_bytes, mb, &ps->full[s], kb * kPBK,
                            b_rows[i]);
        }
    }
    // The copies still in flight land before the CTA may leave.
    for (uint32_t c = g > kPStages ? g - kPStages : 0; c < g; ++c)
        mbar_wait_bounded(&ps->full[c % kPStages], (c / kPStages) & 1u);
}

// Warp 1, one lane: per K block, 4 MMAs of K = 16 into accumulator buffer
// it & 1 (it = the CTA's tile count); a stage is released when its MMAs
// complete, a buffer is announced full when all of the tile's have.
template <int N>
__device__ __forceinline__ void mma_tiles(uint32_t tmem, uint32_t stages, uint32_t stage_bytes,
                                          PipeState *ps, int nk, int n_tiles) {
    constexpr uint32_t idesc = idesc_bf16_f32(kPBM, N);
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
        const int b = it & 1;
        if (it >= 2 && !mbar_wait_bounded(&ps->tempty[b], (uint32_t)((it >> 1) - 1) & 1u)) {
            raise_error(SC_DEV_TIMEOUT);
            ps->abort = 1;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)b * 256u;
        for (int kb = 0; kb < nk; ++kb, ++g) {
            const uint32_t s = g % kPStages;
            if (!mbar_wait_bounded(&ps->full[s], (g / kPStages) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                ps->abort = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t st = stages + s * stage_bytes;
            const uint64_t da = sdesc_k128(st), db = sdesc_k128(st + kPABytes);
#pragma unroll
            for (int j = 0; j < kPBK / 16; ++j)
                mma_bf16(d, da + 2 * j, db + 2 * j, idesc, (kb | j) != 0);
            mma_commit(&ps->empty[s]);
        }
        if (ok) mma_commit(&ps->tfull[b]);
    }
    // No MMA may still write TMEM when it is freed.
    mma_commit(&ps->mma_done);
    mbar_wait_bounded(&ps->mma_done, 0);
}

// Epilogue threads: wait for accumulator buffer b of the CTA's it-th tile.
// The decision to go on is taken together (barrier-OR over the 128 threads),
// so no thread waits at a named barrier the others have left.
__device__ __forceinline__ bool epi_acquire(PipeState *ps, int it) {
    const bool ok = mbar_wait_bounded(&ps->tfull[it & 1], (uint32_t)(it >> 1) & 1u);
    const bool fail = named_or(1, 128, !ok || ps->abort != 0);
    if (!ok) raise_error(SC_DEV_TIMEOUT);
    tc_fence_after();
    return !fail;
}

// Every tcgen05.ld of the buffer has completed (tmem_ld16 waits): release it.
__device__ __forceinline__ void epi_release(PipeState *ps, int it) {
    tc_fence_before();
    mbar_arrive(&ps->tempty[it & 1]);
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *raw) {
    const uint32_t a = smem_addr(raw);
    return raw + (((a + 1023u) & ~1023u) - a);
}

// Shared start of both kernels: barriers, TMEM (2 x 256 columns), PDL wait.
__device__ __forceinline__ uint32_t pipe_start(PipeState *ps, const CUtensorMap *m0,
                                               const CUtensorMap *m1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) pipe_init(ps);
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(m0);
        tma_prefetch_map(m1);
    }
    if (warp == 1) tmem_alloc(&ps->tmem, kPTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ps->tmem;
    pdl_wait();  // inputs may come from the previous kernel in the stream
    pdl_launch_dependents();
    return tmem;
}

__device__ __forceinline__ void pipe_finish(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kPTmemCols);
    }
}

// ------------------------------------------------------------ fused in_proj + conv

template <int K>
__global__ void __launch_bounds__(kPThreads, 1)
    k_in_proj_conv(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                   int64_t T_rows, int D, int H, const bf16 *__restrict__ w,
                   const bf16 *__restrict__ bias, const int32_t *__restrict__ cu, int N,
                   const int32_t *__restrict__ slots, const bf16 *__restrict__ pool, int n_slots,
                   bf16 *__restrict__ y, bf16 *__restrict__ tail, int n_ctiles, int n_tiles) {
    constexpr int OUT = kPBM - (K - 1);  // output rows per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align1024(smem_raw);
    unsigned char *u_tile = base + (size_t)kPStages * kConvStage;
    float *wts = reinterpret_cast<float *>(u_tile + kPBM * kUStride);  // [kConvCh][K]
    float *bsm = wts + kConvCh * 4;
    int32_t *s_cu = reinterpret_cast<int32_t *>(bsm + kConvCh);
    PipeState *ps = reinterpret_cast<PipeState *>(s_cu + kProjCuStaged + 8);
    const uint32_t stages = smem_addr(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / kPBK;
    const uint32_t tmem = pipe_start(ps, &map_h, &map_w);

    if (warp == 0) {
        if (lane == 0)
            produce_tiles<3>(&map_h, &map_w, stages, kConvStage, ps, nk, n_tiles,
                             kConvCh * kPBK * 2, [&](int tile, int &a_row, int (&rows)[3]) {
                                 const int h0 = (tile % n_ctiles) * kConvCh;
                                 a_row = (tile / n_ctiles) * OUT - (K - 1);
                                 rows[0] = h0;
                                 rows[1] = H + h0;
                                 rows[2] = 2 * H + h0;
                             });
    } else if (warp == 1) {
        if (lane == 0) mma_tiles<kConvN>(tmem, stages, kConvStage, ps, nk, n_tiles);
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2..5
        const int et = threadIdx.x - 64;  // 0..127
        const int q = warp & 3;
        const int r = q * 32 + lane;      // tile row = TMEM lane
        // cu_seqlens: staged and checked once per CTA.
        const bool staged = N <= kProjCuStaged;
        bool bad = false;
        for (int j = et; j <= N; j += 128) {
            const int32_t c = cu[j];
            if (staged) s_cu[j] = c;
            if (j == 0 && c != 0) bad = true;
            if (j == N && (int64_t)c != T_rows) bad = true;
            if (j < N && cu[j + 1] < c) bad = true;
        }
        bad = named_or(1, 128, bad);  // also orders the staging above
        if (bad && blockIdx.x == 0 && et == 0) raise_error(SC_DEV_BAD_SEQLENS);
        auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : cu[j]; };
        unsigned char *urow = u_tile + r * kUStride;

        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int h0 = (tile % n_ctiles) * kConvCh;
            const int64_t t = (int64_t)(tile / n_ctiles) * OUT - (K - 1) + r;  // global row
            // This tile's taps and bias (the previous tile is done with them).
            for (int e = et; e < kConvCh * K; e += 128)
                wts[e] = __bfloat162float(w[(int64_t)h0 * K + e]);
            if (bias != nullptr)
                for (int e = et; e < kConvCh; e += 128) bsm[e] = __bfloat162float(bias[h0 + e]);
            if (!epi_acquire(ps, it)) break;
            const uint32_t trow = tmem + (uint32_t)(it & 1) * 256u + ((uint32_t)(q * 32) << 16);

            // Phase A: u = round(round(B) round(x)) of every tile row into u_tile.
            __syncwarp();  // tcgen05.ld is warp-collective: lanes converge first
#pragma unroll
            for (int cc = 0; cc < kConvCh / 16; ++cc) {
                float bv[16], xv[16];
                tmem_ld16(trow + cc * 16, bv);
                tmem_ld16(trow + 2 * kConvCh + cc * 16, xv);
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float u0 =
                        __fmul_rn(Dt<bf16>::round(bv[2 * j]), Dt<bf16>::round(xv[2 * j]));
                    const float u1 = __fmul_rn(Dt<bf16>::round(bv[2 * j + 1]),
                                               Dt<bf16>::round(xv[2 * j + 1]));
                    pk[j] = pack_bf16(u0, u1);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(urow + cc * 32);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            // C of this row, then the buffer goes back to the MMA lane.
            float cv[kConvCh];
#pragma unroll
            for (int cc = 0; cc < kConvCh / 16; ++cc) {
                float tmp[16];
                tmem_ld16(trow + kConvCh + cc * 16, tmp);
#pragma unroll
                for (int j = 0; j < 16; ++j) cv[cc * 16 + j] = Dt<bf16>::round(tmp[j]);
            }
            epi_release(ps, it);
            named_sync(1, 128);  // u_tile, taps and bias complete

            // Phase B: outputs of rows K-1 .. 127 of the tile.
            bool out_row = r >= K - 1 && t < T_rows && !bad;
            int i = 0, slot = 0;
            int64_t s0 = 0, s1 = 0;
            if (out_row) {
                int lo = 0, hi = N - 1;  // the sequence holding row t
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (CU(mid) <= t) lo = mid; else hi = mid - 1;
                }
                i = lo;
                s0 = CU(i);
                s1 = CU(i + 1);
                slot = slots[i];
                if (slot < 0 || slot >= n_slots) {
                    raise_error(SC_DEV_BAD_SLOT);
                    out_row = false;
                }
            }
            if (out_row) {
                const bool fresh_hist = t - s0 >= K - 1;  // whole window inside the sequence
#pragma unroll
                for (int cc = 0; cc < kConvCh / 16; ++cc) {
                    float win[K][16];
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            u_tile + (r - (K - 1) + k) * kUStride + cc * 32);
                        const uint4 a = src[0], b2 = src[1];
                        const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            win[k][2 * j] = bf16_lo(wd[j]);
                            win[k][2 * j + 1] = bf16_hi(wd[j]);
                        }
                    }
                    if (!fresh_hist) {  // window positions before the sequence start: its slot
                        const int64_t rs = t - s0;
#pragma unroll
                        for (int k = 0; k < K; ++k) {
                            const int64_t e = rs + 1 + k;  // index into [state; u_s0 ...]
                            if (e < K)
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    win[k][j] = __bfloat162float(
                                        pool[((int64_t)slot * H + h0 + cc * 16 + j) * K + e]);
                        }
                    }
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        float o[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int c = cc * 16 + j + hh;
                            float z = wts[c * K] * win[0][j + hh];
#pragma unroll
                            for (int k = 1; k < K; ++k) z = fmaf(wts[c * K + k], win[k][j + hh], z);
                            if (bias != nullptr) z = z + bsm[c];
                            o[hh] = cv[c] * z;
                        }
                        pk[j / 2] = pack_bf16(o[0], o[1]);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(y + t * (int64_t)H + h0 + cc * 16);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    if (t >= s1 - K) {  // one of the sequence's last K rows: its u to the tail
                        const int m = (int)(K - (s1 - t));
                        const uint16_t *ur = reinterpret_cast<const uint16_t *>(urow + cc * 32);
                        uint16_t *tl = reinterpret_cast<uint16_t *>(tail);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            tl[((int64_t)i * H + h0 + cc * 16 + j) * K + m] = ur[j];
                    }
                }
            }
            named_sync(1, 128);  // u_tile, taps and bias free for the next tile
        }
    }
    pipe_finish(tmem);
}

// New state of sequence i = the last K entries of [old state; u of its rows]:
// entry m is old[len + m] when len + m < K, else tail[i][h][m]. One thread per
// (sequence, 8 channels); nothing for empty sequences.
template <int K>
__global__ void __launch_bounds__(256)
    k_commit_states(const int32_t *__restrict__ cu, int N, int64_t T_rows,
                    const int32_t *__restrict__ slots, const uint16_t *__restrict__ tail,
                    uint16_t *__restrict__ pool, int n_slots, int H) {
    pdl_wait();
    pdl_launch_dependents();
    int bad = 0;
    for (int j = threadIdx.x; j <= N; j += blockDim.x) {
        const int32_t c = cu[j];
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && cu[j + 1] < c) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(SC_DEV_BAD_SEQLENS);
        return;
    }
    const int groups = H / kCh;
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (unit >= (int64_t)N * groups) return;
    const int i = (int)(unit / groups), h = (int)(unit % groups) * kCh;
    const int64_t len = (int64_t)cu[i + 1] - cu[i];
    if (len == 0) return;
    const int slot = slots[i];
    if (slot < 0 || slot >= n_slots) {
        if (h == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
        uint16_t *st = pool + ((int64_t)slot * H + h + c) * K;
        const uint16_t *tl = tail + ((int64_t)i * H + h + c) * K;
        uint16_t old[K], nw[K];
#pragma unroll
        for (int k = 0; k < K; ++k) old[k] = st[k];
#pragma unroll
        for (int m = 0; m < K; ++m) nw[m] = len + m < K ? old[len + m] : tl[m];
#pragma unroll
        for (int m = 0; m < K; ++m) st[m] = nw[m];
    }
}

// ------------------------------------------------------------ out_proj

__global__ void __launch_bounds__(kPThreads, 1)
    k_out_proj(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               int64_t M_rows, int Kdim, int N_cols, bf16 *__restrict__ out, int n_ntiles,
               int n_tiles) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align1024(smem_raw);
    PipeState *ps = reinterpret_cast<PipeState *>(base + (size_t)kPStages * kOutStage);
    const uint32_t stages = smem_addr(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = Kdim / kPBK;
    const uint32_t tmem = pipe_start(ps, &map_a, &map_b);

    if (warp == 0) {
        if (lane == 0)
            produce_tiles<1>(&map_a, &map_b, stages, kOutStage, ps, nk, n_tiles,
                             kOutN * kPBK * 2, [&](int tile, int &a_row, int (&rows)[1]) {
                                 a_row = (tile / n_ntiles) * kPBM;
                                 rows[0] = (tile % n_ntiles) * kOutN;
                             });
    } else if (warp == 1) {
        if (lane == 0) mma_tiles<kOutN>(tmem, stages, kOutStage, ps, nk, n_tiles);
        __syncwarp();
    } else {
        const int q = warp & 3;
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int64_t t = (int64_t)(tile / n_ntiles) * kPBM + q * 32 + lane;
            const int col0 = (tile % n_ntiles) * kOutN;
            if (!epi_acquire(ps, it)) break;
            const uint32_t trow = tmem + (uint32_t)(it & 1) * 256u + ((uint32_t)(q * 32) << 16);
            const bool store = t < M_rows;
#pragma unroll 1
            for (int cc = 0; cc < kOutN / 16; ++cc) {
                __syncwarp();
                float v[16];
                tmem_ld16(trow + cc * 16, v);
                if (!store) continue;
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) pk[j] = pack_bf16(v[2 * j], v[2 * j + 1]);
                uint4 *dst = reinterpret_cast<uint4 *>(out + t * (int64_t)N_cols + col0 + cc * 16);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            __syncwarp();
            epi_release(ps, it);
        }
    }
    pipe_finish(tmem);
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A row-major bf16 matrix [outer, inner] read in {64, box_rows} boxes with
// the 128-byte swizzle; rows past the end (or before row 0) read as zeros.
static cudaError_t map_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
                          uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kPBK, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Opt a kernel in to its dynamic shared memory once per device.
template <typename F>
static cudaError_t smem_opt_in(F kern, size_t bytes, std::atomic<unsigned long long> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && (done.load() & (1ull << dev))) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev < 64) done.fetch_or(1ull << dev);
    return e;
}

size_t in_proj_workspace_bytes(int H, int K, int N) { return (size_t)N * H * K * 2; }

template <int K>
static cudaError_t in_proj_inst(const CUtensorMap &mh, const CUtensorMap &mw, int64_t T, int D,
                                int H, const void *w, const void *bias, const int32_t *cu, int N,
                                const int32_t *slots, void *pool, int n_slots, void *y,
                                void *tail, int sm_count, cudaStream_t stream) {
    constexpr int OUT = kPBM - (K - 1);
    cudaError_t e;
    if (T > 0) {
        static std::atomic<unsigned long long> done{0};
        e = smem_opt_in(k_in_proj_conv<K>, conv_smem_bytes(), done);
        if (e != cudaSuccess) return e;
        const int n_ctiles = H / kConvCh;
        const int64_t n_tiles = (T + OUT - 1) / OUT * n_ctiles;
        const int grid = (int)(n_tiles < sm_count ? n_tiles : sm_count);  // persistent
        e = launch_pdl(k_in_proj_conv<K>, dim3((unsigned)grid), dim3(kPThreads),
                       conv_smem_bytes(), stream, mh, mw, T, D, H, (const bf16 *)w,
                       (const bf16 *)bias, cu, N, slots, (const bf16 *)pool, n_slots, (bf16 *)y,
                       (bf16 *)tail, n_ctiles, (int)n_tiles);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = (int64_t)N * (H / kCh);
    if (units == 0) return cudaSuccess;
    return launch_pdl(k_commit_states<K>, dim3((unsigned)((units + 255) / 256)), dim3(256), 0,
                      stream, cu, N, T, slots, (const uint16_t *)tail, (uint16_t *)pool, n_slots,
                      H);
}

cudaError_t launch_in_proj_prefill(int D, int H, int K, const void *hidden, int64_t T,
                                   const void *w_in, const void *w, const void *bias,
                                   const int32_t *cu, int N, const int32_t *slots, void *pool,
                                   int n_slots, void *y, void *workspace, int sm_count,
                                   cudaStream_t stream) {
    CUtensorMap mh, mw;
    if (T > 0) {
        cudaError_t e = map_2d(&mh, hidden, (uint64_t)D, (uint64_t)T, kPBM);
        if (e != cudaSuccess) return e;
        e = map_2d(&mw, w_in, (uint64_t)D, (uint64_t)3 * H, kConvCh);
        if (e != cudaSuccess) return e;
    }
    switch (K) {
        case 1: return in_proj_inst<1>(mh, mw, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        case 2: return in_proj_inst<2>(mh, mw, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        case 3: return in_proj_inst<3>(mh, mw, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        default: return in_proj_inst<4>(mh, mw, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
    }
}

cudaError_t launch_out_proj(int H, int D, const void *y, int64_t T, const void *w_out, void *out,
                            int sm_count, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    CUtensorMap ma, mb;
    cudaError_t e = map_2d(&ma, y, (uint64_t)H, (uint64_t)T, kPBM);
    if (e != cudaSuccess) return e;
    e = map_2d(&mb, w_out, (uint64_t)H, (uint64_t)D, kOutN);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> done{0};
    e = smem_opt_in(k_out_proj, out_smem_bytes(), done);
    if (e != cudaSuccess) return e;
    const int n_ntiles = D / kOutN;
    const int64_t n_tiles = (T + kPBM - 1) / kPBM * n_ntiles;
    const int grid = (int)(n_tiles < sm_count ? n_tiles : sm_count);  // persistent
    return launch_pdl(k_out_proj, dim3((unsigned)grid), dim3(kPThreads), out_smem_bytes(), stream,
                      ma, mb, T, H, D, (bf16 *)out, n_ntiles, (int)n_tiles);
}

cudaError_t take_error_proj(cudaStream_t stream, unsigned int *code) {
    return take_error_here(stream, code);
}

}  // namespace sc
