// proj.cu -- the ShortConv layer's projections on the tcgen05 tensor cores.
//
// The MAX LFM2 article (section "短卷积实现（LFM2ShortConv）") gives the layer:
// in_proj maps the hidden state to three parts b, c, xv; bx = b * xv goes
// through the causal depthwise conv; c * conv_out goes through out_proj.
//
// k_in_proj_conv fuses everything up to out_proj into the in_proj GEMM: a CTA
// pair computes the [B | C | x] product block of 128 channels for 2 x 128
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
// writes the new states: no tile writes a slot another tile reads. A call
// with one sequence skips that pass: its walk gives each column's first and
// last row tiles to one cluster, and the CTA with the last one writes the
// new state after the cluster's final barrier (see TileWalk::group).
//
// k_out_proj is the plain out_proj GEMM (256 x 256 tiles a pair) on the same
// mainloop; its epilogue rounds to bf16 into swizzled shared-memory boxes
// that TMA copies store.
//
// Warp roles: warp 0 issues the TMA copies, warp 1 owns the TMEM allocation
// and one of its lanes issues the MMAs, the other warps run the epilogue
// (warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31): 8 epilogue warps in
// the fused kernel, two per lane quarter with 32 channels each, so the conv
// epilogue keeps pace with the tensor cores; 4 in out_proj. Every mbarrier
// wait gives up after 2 s (SC_DEV_TIMEOUT); the TMEM is always freed.
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

constexpr int kPBM = 128;                     // rows per CTA tile = TMEM lanes
constexpr int kPBK = 64;                      // K per stage: one 128-byte swizzle row
constexpr int kOutThreads = 192;              // producer, MMA and 4 epilogue warps
constexpr uint32_t kPABytes = kPBM * kPBK * 2;  // 16 KB

#ifndef SC_PROJ_CLUSTER
#define SC_PROJ_CLUSTER 2  // 2: CTA pairs run 256-row MMAs (cta_group::2); 1: single CTAs
#endif
#ifndef SC_INPROJ_STAGES
#define SC_INPROJ_STAGES 4  // stage ring depth of the fused in_proj (40 KB a stage)
#endif
#ifndef SC_OUTPROJ_STAGES
#define SC_OUTPROJ_STAGES (SC_PROJ_CLUSTER == 2 ? 6 : 4)  // stage ring depth, out_proj
#endif
constexpr int kPCluster = SC_PROJ_CLUSTER;
constexpr uint32_t kPTmemCols = 512;  // all of TMEM: accumulator buffers of 256 columns
constexpr int kInStages = SC_INPROJ_STAGES;
constexpr int kOutStages = SC_OUTPROJ_STAGES;
constexpr int kMaxStages = 8;
static_assert(kPCluster == 1 || kPCluster == 2, "CTA pairs or single CTAs");

// Fused tile: the B | C | x product columns of kConvCh channels, laid out in
// TMEM as [B | C | x] (column c, kConvCh + c, 2 kConvCh + c for channel c).
// CTA pairs: 128 channels, one N = 256 MMA (B | C) into columns 0.. and one
// N = 128 MMA (x) into columns 256..; 384 columns, one accumulator buffer.
// Single CTAs: 64 channels, one N = 192 MMA; two buffers of 256 columns.
// Either way a CTA stages A and three 64-row boxes of w_in (40 KB a stage).
constexpr int kConvCh = kPCluster == 2 ? 128 : 64;
constexpr int kConvN1 = kPCluster == 2 ? 256 : 192;   // first MMA's N
constexpr int kConvN2 = kPCluster == 2 ? 128 : 0;     // second MMA's N (0: none)
constexpr int kInBufs = kPCluster == 2 ? 1 : 2;       // accumulator buffers
constexpr int kConvBoxRows = 64;
constexpr uint32_t kConvBox = kConvBoxRows * kPBK * 2;   // 8 KB
constexpr uint32_t kConvStage = kPABytes + 3 * kConvBox;  // 40 KB
constexpr int kOutBufs = 2;
constexpr int kUStride = kConvCh * 2 + 16;    // bytes per u row (+16: conflict-free)
constexpr int kProjCuStaged = 512;
#ifndef SC_INPROJ_EPI_WARPS
#define SC_INPROJ_EPI_WARPS 8  // epilogue warps of the fused kernel: 4 or 8
#endif
// Epilogue warp w reads TMEM lanes 32 (w % 4) ..; with 8 warps two share each
// lane quarter and each takes half of the tile's channels.
constexpr int kInEpiWarps = SC_INPROJ_EPI_WARPS;
constexpr int kInEpiThreads = 32 * kInEpiWarps;
constexpr int kInThreads = 64 + kInEpiThreads;
constexpr int kChPerWarp = kConvCh * 4 / kInEpiWarps;  // channels per epilogue warp
constexpr uint32_t kInYBox = 32 * kPBK * 2;  // a y box: 32 rows x 64 channels, 4 KB
#ifndef SC_INPROJ_YBOX
#define SC_INPROJ_YBOX 1
#endif
constexpr bool kInYBoxed = SC_INPROJ_YBOX && kChPerWarp == kPBK;  // a warp's channels fill one y box
constexpr int kChPass = 32;  // channels of one TMEM read pass (3 x 32 registers in flight)
static_assert(kInEpiWarps == 4 || kInEpiWarps == 8, "4 or 8 epilogue warps");

constexpr int kOutN = 256;                    // out_proj N per tile
constexpr int kOutBoxRows = kOutN / kPCluster;
constexpr uint32_t kOutBox = kOutBoxRows * kPBK * 2;
constexpr uint32_t kOutStage = kPABytes + kOutBox;  // 48 KB single, 32 KB a pair CTA
// out_proj's store staging: per epilogue warp two boxes of 32 rows x 64
// columns (128-byte swizzle), filled from TMEM and written by TMA stores.
constexpr uint32_t kOutStgBox = 32 * kPBK * 2;  // 4 KB
constexpr uint32_t kOutStg = 4 * 2 * kOutStgBox;  // 32 KB
constexpr int kOutBoxes = kOutN / kPBK;           // boxes of a warp's tile rows
static_assert(4u * kOutBoxes * kOutStgBox <= (uint32_t)kOutStages * kOutStage,
              "the stage ring holds a whole tile's boxes");
// Shared memory after the stage ring: barriers and flags. The accumulator
// is double-buffered in TMEM (columns 0.. and 256..): the MMA lane fills one
// buffer while the epilogue warps drain the other.
struct PipeState {
    uint64_t full[kMaxStages];   // stage loaded (TMA bytes)
    uint64_t empty[kMaxStages];  // stage consumed (MMA commit)
    uint64_t tfull[2];         // accumulator buffer ready (MMA commit)
    uint64_t tempty[2];        // accumulator buffer drained (128 epilogue threads)
    uint64_t mma_done;         // every MMA of this CTA completed
    uint32_t tmem;
    volatile int abort;        // set by the producer or the MMA lane when a wait gave up
};

constexpr size_t kConvExtra = (size_t)kPBM * kUStride          // u tile
                              + kConvCh * 4 * sizeof(float)    // taps, tap-major
                              + kConvCh * sizeof(float)        // bias
                              + (kProjCuStaged + 8) * 4;       // staged cu_seqlens
constexpr size_t conv_smem_bytes() {
    return 1024 + (size_t)kInStages * kConvStage + kConvExtra + sizeof(PipeState);
}
constexpr size_t out_smem_bytes() {
    return 1024 + (size_t)kOutStages * kOutStage + kOutStg + sizeof(PipeState);
}
static_assert(conv_smem_bytes() <= 232448 && out_smem_bytes() <= 232448,
              "stage ring larger than a CTA's shared memory");
static_assert(kInStages <= kMaxStages && kOutStages <= kMaxStages, "too many stages");
static_assert(kInEpiWarps * kInYBox <= (uint32_t)kInStages * kConvStage,
              "the stage ring holds every epilogue warp's y box");

// ------------------------------------------------------------ persistent mainloop
//
// CL = 1: one CTA runs 128-row MMAs (cta_group::1). CL = 2: the two CTAs of a
// cluster run 256-row MMAs as a pair (cta_group::2): each stages its own 128
// rows of A and half of B's N rows, the leader (rank 0) issues the MMAs, and
// each CTA's TMEM receives its own rows of the result. Per SM that halves the
// B bytes staged and read by the tensor core. The CTAs of a cluster take CL
// consecutive row tiles of one column tile; clusters walk the tile groups c,
// c + n_clusters, ...; the stage ring runs on across tiles (k-block counter g
// over all of the CTA's tiles).

struct TileWalk {
    int first, step, n_groups, rank, CL;
    int single_cols, pairs;  // single-sequence schedule: column tiles (0: off), row-tile pairs

    // Single-sequence schedule of the fused prefill (one sequence over several
    // row-tile pairs): walk position i -> tile group. Positions 0 .. C-1 take
    // each column's first pair, and the last position of each of those
    // clusters takes the same column's last pair: the cluster that reads a
    // column's old state (its first rows) also writes the new one (its last
    // rows), after all of its other tiles. The other positions take the
    // middle pairs in order. Needs C <= clusters and n_groups >= clusters + C.
    __device__ __forceinline__ int group(int i) const {
        const int C = single_cols;
        if (i < C) return i;
        const int L0 = (n_groups - 1) / step, r0 = (n_groups - 1) % step;
        auto last_of = [&](int c) { return c + step * (c <= r0 ? L0 : L0 - 1); };
        const int c = i % step;
        if (c < C && i == last_of(c)) return (pairs - 1) * C + c;
        int below = C;  // special positions before i
        for (int k = 0; k < C; ++k) below += last_of(k) < i ? 1 : 0;
        return C + (i - below);
    }
    // Row tile and column tile of the tile at walk position pos for this CTA.
    __device__ __forceinline__ void at(int pos, int n_col_tiles, int &mt, int &ct) const {
        const int grp = single_cols ? group(pos) : pos;
        ct = grp % n_col_tiles;
        mt = (grp / n_col_tiles) * CL + rank;
    }
};

template <int CL>
__device__ __forceinline__ TileWalk tile_walk(int n_row_tiles, int n_col_tiles,
                                              bool single = false) {
    TileWalk w;
    w.CL = CL;
    w.rank = CL > 1 ? (int)cluster_ctarank() : 0;
    w.first = blockIdx.x / CL;
    w.step = gridDim.x / CL;
    w.pairs = (n_row_tiles + CL - 1) / CL;
    w.n_groups = w.pairs * n_col_tiles;
    // With one pair every group is its column's first and last: no reordering.
    w.single_cols = single && w.pairs > 1 ? n_col_tiles : 0;
    return w;
}

__device__ __forceinline__ void pipe_init(PipeState *ps, int CL, int epi_warps) {
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) {
        mbar_init(&ps->full[s], 1);   // the (leader's) producer; bytes of both CTAs
        mbar_init(&ps->empty[s], 1);  // the (leader's) MMA commit
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        mbar_init(&ps->tfull[b], 1);
        mbar_init(&ps->tempty[b], epi_warps * CL);  // one lane per epilogue warp of each CTA
    }
    mbar_init(&ps->mma_done, 1);
    ps->abort = 0;
    mbar_fence_init();
}

// Warp 0, one lane. coords(mt, ct, a_row, rows) gives the tile's A row and the
// first rows of this CTA's NB boxes of B (box_bytes each); a stage holds A,
// then the boxes.
template <int S, int NB, int CL, typename Coords>
__device__ __forceinline__ void produce_tiles(const CUtensorMap *ma, const CUtensorMap *mb,
                                              uint32_t stages, uint32_t stage_bytes,
                                              PipeState *ps, int nk, const TileWalk &tw,
                                              int n_col_tiles, uint32_t box_bytes,
                                              Coords coords) {
    const bool leader = tw.rank == 0;
    uint32_t g = 0;
    bool ok = true;
    for (int grp = tw.first; grp < tw.n_groups && ok; grp += tw.step) {
        int mt, ct, a_row, rows[NB];
        tw.at(grp, n_col_tiles, mt, ct);
        coords(mt, ct, a_row, rows);
        for (int kb = 0; kb < nk; ++kb, ++g) {
            const uint32_t s = g % S;
            if (g >= S && !mbar_wait_bounded(&ps->empty[s], (g / S - 1) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                ps->abort = 1;
                ok = false;
                break;
            }
            const uint32_t st = stages + s * stage_bytes;
            if constexpr (CL == 1) {
                mbar_arrive_expect_tx(&ps->full[s], stage_bytes);
                tma_load_2d(st, ma, &ps->full[s], kb * kPBK, a_row);
#pragma unroll
                for (int i = 0; i < NB; ++i)
                    tma_load_2d(st + kPABytes + i * box_bytes, mb, &ps->full[s], kb * kPBK,
                                rows[i]);
            } else {  // both CTAs' bytes count on the leader's barrier
                const uint32_t bar = cluster_map(smem_addr(&ps->full[s]), 0);
                if (leader) mbar_arrive_expect_tx(&ps->full[s], 2 * stage_bytes);
                tma_load_2d_pair(st, ma, bar, kb * kPBK, a_row);
#pragma unroll
                for (int i = 0; i < NB; ++i)
                    tma_load_2d_pair(st + kPABytes + i * box_bytes, mb, bar, kb * kPBK, rows[i]);
            }
        }
    }
    // The copies in flight land before the CTA may leave (the leader's barrier
    // counts both CTAs' bytes), and so do the MMA-commit arrivals that release
    // the last stages.
    if (CL == 1 || leader)
        for (uint32_t c = g > S ? g - S : 0; c < g; ++c)
            mbar_wait_bounded(&ps->full[c % S], (c / S) & 1u);
    if (ok)
        for (uint32_t c = g > S ? g - S : 0; c < g; ++c)
            mbar_wait_bounded(&ps->empty[c % S], (c / S) & 1u);
}

// Warp 1, one lane of the (leader) CTA: per 16-deep K step one MMA of N1
// columns (B rows 0 .. N1/CL - 1 of the CTA's stage) into the buffer's
// columns 0.., and, if N2 > 0, one of N2 columns (the next N2/CL B rows)
// into columns C2..; into accumulator buffer it % NBUF (it = the CTA's tile
// count, buffers BS columns apart). A stage is released when its MMAs
// complete, a buffer is announced full when all of the tile's have.
template <int S, int N1, int N2, int CL, int NBUF, int C2 = 256, int BS = 256>
__device__ __forceinline__ void mma_tiles(uint32_t tmem, uint32_t stages, uint32_t stage_bytes,
                                          PipeState *ps, int nk, const TileWalk &tw) {
    static_assert(C2 >= N1 && (N2 == 0 || C2 + N2 <= BS || NBUF == 1),
                  "the MMAs of one buffer do not overlap each other or the next buffer");
    static_assert((NBUF - 1) * BS + (N2 > 0 ? C2 + N2 : N1) <= (int)kPTmemCols, "fits TMEM");
    constexpr uint32_t idesc1 = idesc_bf16_f32(kPBM * CL, N1);
    constexpr uint32_t idesc2 = idesc_bf16_f32(kPBM * CL, N2 > 0 ? N2 : 16);
    constexpr uint32_t b2_off = (uint32_t)(N1 / CL) * kPBK * 2;  // bytes to the second B part
    constexpr uint16_t both = 3;
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (int grp = tw.first; grp < tw.n_groups && ok; grp += tw.step, ++it) {
        const int b = it % NBUF, use = it / NBUF;
        if (use >= 1 && !mbar_wait_bounded(&ps->tempty[b], (uint32_t)(use - 1) & 1u)) {
            raise_error(SC_DEV_TIMEOUT);
            ps->abort = 1;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)b * (uint32_t)BS;  // NBUF == 1: b == 0
        for (int kb = 0; kb < nk; ++kb, ++g) {
            const uint32_t s = g % S;
            if (!mbar_wait_bounded(&ps->full[s], (g / S) & 1u)) {
                raise_error(SC_DEV_TIMEOUT);
                ps->abort = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t st = stages + s * stage_bytes;
            const uint64_t da = sdesc_k128(st), db = sdesc_k128(st + kPABytes);
            const uint64_t db2 = sdesc_k128(st + kPABytes + b2_off);
#pragma unroll
            for (int j = 0; j < kPBK / 16; ++j) {
                const uint32_t acc = (kb | j) != 0;
                if constexpr (CL == 1) {
                    mma_bf16(d, da + 2 * j, db + 2 * j, idesc1, acc);
                    if constexpr (N2 > 0) mma_bf16(d + C2, da + 2 * j, db2 + 2 * j, idesc2, acc);
                } else {
                    mma_bf16_pair(d, da + 2 * j, db + 2 * j, idesc1, acc);
                    if constexpr (N2 > 0)
                        mma_bf16_pair(d + C2, da + 2 * j, db2 + 2 * j, idesc2, acc);
                }
            }
            if constexpr (CL == 1)
                mma_commit(&ps->empty[s]);
            else
                mma_commit_pair(&ps->empty[s], both);  // the stage of both CTAs
        }
        if (ok) {
            if constexpr (CL == 1)
                mma_commit(&ps->tfull[b]);
            else
                mma_commit_pair(&ps->tfull[b], both);
        }
    }
    // No MMA may still write TMEM when it is freed.
    if constexpr (CL == 1)
        mma_commit(&ps->mma_done);
    else
        mma_commit_pair(&ps->mma_done, 1);
    mbar_wait_bounded(&ps->mma_done, 0);
}

// Epilogue threads: wait for the accumulator buffer of the CTA's it-th tile.
// The decision to go on is taken together (barrier-OR over the 128 threads),
// so no thread waits at a named barrier the others have left.
template <int NBUF>
__device__ __forceinline__ bool epi_acquire(PipeState *ps, int it, int epi_threads) {
    const bool ok = mbar_wait_bounded(&ps->tfull[it % NBUF], (uint32_t)(it / NBUF) & 1u);
    const bool fail = named_or(1, epi_threads, !ok || ps->abort != 0);
    if (!ok) raise_error(SC_DEV_TIMEOUT);
    tc_fence_after();
    return !fail;
}

// Every tcgen05.ld of the buffer has completed (tmem_ld16 waits): one lane
// per warp releases it on the (leader's) barrier.
template <int CL, int NBUF>
__device__ __forceinline__ void epi_release(PipeState *ps, int it, int rank) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        uint64_t *bar = &ps->tempty[it % NBUF];
        if (CL == 1 || rank == 0)
            mbar_arrive(bar);
        else
            mbar_arrive_cluster(cluster_map(smem_addr(bar), 0));
    }
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *raw) {
    const uint32_t a = smem_addr(raw);
    return raw + (((a + 1023u) & ~1023u) - a);
}

// Shared start of both kernels: barriers, TMEM, PDL wait; with pairs, no CTA
// goes on before every CTA's barriers exist.
template <int CL>
__device__ __forceinline__ uint32_t pipe_start(PipeState *ps, const CUtensorMap *m0,
                                               const CUtensorMap *m1, int epi_warps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) pipe_init(ps, CL, epi_warps);
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(m0);
        tma_prefetch_map(m1);
    }
    if (warp == 1) {
        if constexpr (CL == 1)
            tmem_alloc(&ps->tmem, kPTmemCols);
        else
            tmem_alloc_pair(&ps->tmem, kPTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (CL > 1) cluster_sync();
    const uint32_t tmem = ps->tmem;
    pdl_wait();  // inputs may come from the previous kernel in the stream
    pdl_launch_dependents();
    return tmem;
}

// With pairs, no CTA leaves while the other may still write its shared
// memory or arrive on its barriers; the pair frees its TMEM together.
template <int CL>
__device__ __forceinline__ void pipe_finish(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if constexpr (CL > 1) cluster_sync();
    if ((threadIdx.x >> 5) == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (CL == 1)
            tmem_dealloc(tmem, kPTmemCols);
        else
            tmem_dealloc_pair(tmem, kPTmemCols);
    }
}

// ------------------------------------------------------------ fused in_proj + conv

template <int K, int CL>
__global__ void __launch_bounds__(kInThreads, 1)
    k_in_proj_conv(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                   const __grid_constant__ CUtensorMap map_y,
                   int64_t T_rows, int D, int H, const bf16 *__restrict__ w,
                   const bf16 *__restrict__ bias, const int32_t *__restrict__ cu, int N,
                   const int32_t *__restrict__ slots, bf16 *__restrict__ pool, int n_slots,
                   bf16 *__restrict__ y, bf16 *__restrict__ tail, int n_ctiles, int n_mtiles,
                   int single) {
    constexpr int OUT = kPBM - (K - 1);  // output rows per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align1024(smem_raw);
    unsigned char *u_tile = base + (size_t)kInStages * kConvStage;
    float *wts = reinterpret_cast<float *>(u_tile + kPBM * kUStride);  // [kConvCh][K]
    float *bsm = wts + kConvCh * 4;
    int32_t *s_cu = reinterpret_cast<int32_t *>(bsm + kConvCh);
    PipeState *ps = reinterpret_cast<PipeState *>(s_cu + kProjCuStaged + 8);
    const uint32_t stages = smem_addr(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / kPBK;
    const uint32_t tmem = pipe_start<CL>(ps, &map_h, &map_w, kInEpiWarps);
    const TileWalk tw = tile_walk<CL>(n_mtiles, n_ctiles, single != 0);
    // Single-sequence schedule: the CTA's last tile, and whether every tile ran.
    int fin_mt = -1, fin_ct = 0;
    bool fin_ok = false;

    if (warp == 0) {
        auto conv_coords = [&](int mt, int ct, int &a_row, int (&rows)[3]) {
            const int h0 = ct * kConvCh;
            a_row = mt * OUT - (K - 1);
            if constexpr (CL == 2) {
                // First MMA's B rows (B | C of 128 channels): rank 0 holds the
                // 128 of B, rank 1 the 128 of C; second MMA's (x): 64 each.
                rows[0] = tw.rank * H + h0;
                rows[1] = tw.rank * H + h0 + 64;
                rows[2] = 2 * H + h0 + 64 * tw.rank;
            } else {  // B | C | x of 64 channels
#pragma unroll
                for (int i = 0; i < 3; ++i) rows[i] = i * H + h0;
            }
        };
        if (lane == 0)
            produce_tiles<kInStages, 3, CL>(
                &map_h, &map_w, stages, kConvStage, ps, nk, tw, n_ctiles, kConvBox, conv_coords);
    } else if (warp == 1) {
        if (lane == 0 && tw.rank == 0)
            mma_tiles<kInStages, kConvN1, kConvN2, CL, kInBufs>(tmem, stages, kConvStage, ps, nk,
                                                                 tw);
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2 .. 2 + kInEpiWarps - 1
        const int et = threadIdx.x - 64;        // 0 .. kInEpiThreads - 1
        const int q = warp & 3;                 // TMEM lane quarter
        const int r = q * 32 + lane;            // tile row = TMEM lane
        const int cw = ((warp - 2) >> 2) * kChPerWarp;  // this warp's first channel
        // cu_seqlens: staged and checked once per CTA.
        const bool staged = N <= kProjCuStaged;
        bool bad = false;
        for (int j = et; j <= N; j += kInEpiThreads) {
            const int32_t c = gld(cu + j);
            if (staged) s_cu[j] = c;
            if (j == 0 && c != 0) bad = true;
            if (j == N && (int64_t)c != T_rows) bad = true;
            if (j < N && gld(cu + j + 1) < c) bad = true;
        }
        bad = named_or(1, kInEpiThreads, bad);  // also orders the staging above
        if (bad && blockIdx.x == 0 && et == 0) raise_error(SC_DEV_BAD_SEQLENS);
        auto CU = [&](int j) -> int64_t { return staged ? s_cu[j] : gld(cu + j); };
        unsigned char *urow = u_tile + r * kUStride;
        // The last tile's y box of this warp (32 rows x 64 channels) in the stage ring.
        unsigned char *ybox = base + (size_t)(warp - 2) * kInYBox;
        if (et == 0) tma_prefetch_map(&map_y);

        int it = 0;
        bool all = true;
        for (int grp = tw.first; grp < tw.n_groups; grp += tw.step, ++it) {
            int mt, ct;
            tw.at(grp, n_ctiles, mt, ct);
            fin_mt = mt;
            fin_ct = ct;
            const int h0 = ct * kConvCh;
            const int64_t t = (int64_t)mt * OUT - (K - 1) + r;  // global row (past T: no output)
            // This tile's taps (tap-major: wts[k * 64 + c]) and bias; the previous
            // tile is done with them.
            // (With H % 128 == 64 the last column tile is half full: its upper 64
            // channels are computed from other weight rows or zeros, never stored.)
            for (int e = et; e < kConvCh * K; e += kInEpiThreads)
                wts[(e % K) * kConvCh + e / K] =
                    h0 + e / K < H ? __bfloat162float(gld(w + (int64_t)h0 * K + e)) : 0.f;
            if (bias != nullptr)
                for (int e = et; e < kConvCh; e += kInEpiThreads)
                    bsm[e] = h0 + e < H ? __bfloat162float(gld(bias + h0 + e)) : 0.f;
            if (!epi_acquire<kInBufs>(ps, it, kInEpiThreads)) {
                all = false;
                break;
            }
            const uint32_t trow =
                tmem + (uint32_t)(it % kInBufs) * 256u + ((uint32_t)(q * 32) << 16) + cw;

            // Phase A: this warp's channels in passes of kChPass, each pass with its
            // B, x and C loads in flight at once. Each pass only packs: B and x to
            // bf16 pairs, u = round(B x) by one bf16x2 multiply (the exact product
            // rounded once), C to bf16 pairs. The accumulator buffer goes back to
            // the MMA lane after the last pass; u then goes to u_tile.
            uint32_t up[kChPerWarp / 2], cvp[kChPerWarp / 2];  // two channels a register
            __syncwarp();  // tcgen05.ld is warp-collective: lanes converge first
#pragma unroll
            for (int p0 = 0; p0 < kChPerWarp; p0 += kChPass) {
                constexpr int NC = kChPass / 16;
                uint32_t rb[NC][16], rx[NC][16], rc[NC][16];
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    const uint32_t col = trow + p0 + cc * 16;
                    tmem_ld16_nowait(col, rb[cc]);
                    tmem_ld16_nowait(col + 2 * kConvCh, rx[cc]);
                    tmem_ld16_nowait(col + kConvCh, rc[cc]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    tmem_regs_ready(rb[cc]);
                    tmem_regs_ready(rx[cc]);
                    tmem_regs_ready(rc[cc]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int e = (p0 + cc * 16) / 2 + j;
                        up[e] = bf2_mul(pack_bf16(__uint_as_float(rb[cc][2 * j]),
                                                  __uint_as_float(rb[cc][2 * j + 1])),
                                        pack_bf16(__uint_as_float(rx[cc][2 * j]),
                                                  __uint_as_float(rx[cc][2 * j + 1])));
                        cvp[e] = pack_bf16(__uint_as_float(rc[cc][2 * j]),
                                           __uint_as_float(rc[cc][2 * j + 1]));
                    }
                }
            }
            epi_release<CL, kInBufs>(ps, it, tw.rank);  // the accumulator buffer is read
#pragma unroll
            for (int e = 0; e < kChPerWarp / 2; e += 4)
                *reinterpret_cast<uint4 *>(urow + (cw + 2 * e) * 2) =
                    make_uint4(up[e], up[e + 1], up[e + 2], up[e + 3]);
            named_sync(1, kInEpiThreads);  // u_tile, taps and bias complete

            // Phase B: outputs of rows K-1 .. 127 of the tile, this warp's channels.
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
                slot = gld(slots + i);
                if (slot < 0 || slot >= n_slots) {
                    raise_error(SC_DEV_BAD_SLOT);
                    out_row = false;
                }
            }
            // The CTA's last tile: its MMAs have consumed every stage and no load
            // follows, so the warp's 32 rows x 64 channels go out as one TMA box
            // (128-byte swizzle) when each of its rows is an output row or past
            // the end; a box with a history row (the previous tile's output) or a
            // refused row takes the 16-byte stores.
            const int64_t box_row = (int64_t)mt * OUT - (K - 1) + q * 32;
            const bool boxed = kInYBoxed && grp + tw.step >= tw.n_groups && box_row >= 0 &&
                               __all_sync(0xffffffffu, out_row || t >= T_rows);
            if (out_row) {
                const bool fresh_hist = t - s0 >= K - 1;  // whole window inside the sequence
#pragma unroll
                for (int sc8 = 0; sc8 < kChPerWarp / 8; ++sc8) {  // 8-channel sub-chunks
                    const int c0 = cw + sc8 * 8;  // first channel of the sub-chunk in the tile
                    if (h0 + c0 >= H) break;      // past the last channel (H % 64 == 0)
                    float win[K][8], wk[K][8], bv[8];
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(
                            u_tile + (r - (K - 1) + k) * kUStride + c0 * 2);
                        const uint32_t wd[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            win[k][2 * j] = bf16_lo(wd[j]);
                            win[k][2 * j + 1] = bf16_hi(wd[j]);
                        }
                        const float4 *tp = reinterpret_cast<const float4 *>(wts + k * kConvCh + c0);
                        const float4 t0 = tp[0], t1 = tp[1];
                        wk[k][0] = t0.x; wk[k][1] = t0.y; wk[k][2] = t0.z; wk[k][3] = t0.w;
                        wk[k][4] = t1.x; wk[k][5] = t1.y; wk[k][6] = t1.z; wk[k][7] = t1.w;
                    }
                    if (bias != nullptr) {
                        const float4 *bp = reinterpret_cast<const float4 *>(bsm + c0);
                        const float4 b0 = bp[0], b1 = bp[1];
                        bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
                        bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
                    }
                    if (!fresh_hist) {  // window positions before the sequence start: its slot
                        const int64_t rs = t - s0;
#pragma unroll
                        for (int k = 0; k < K; ++k) {
                            const int64_t e = rs + 1 + k;  // index into [state; u_s0 ...]
                            if (e < K)
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    win[k][j] = __bfloat162float(
                                        gld(pool + ((int64_t)slot * H + h0 + c0 + j) * K + e));
                        }
                    }
                    uint32_t pk[4];
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        float o[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            float z = wk[0][j + hh] * win[0][j + hh];
#pragma unroll
                            for (int k = 1; k < K; ++k) z = fmaf(wk[k][j + hh], win[k][j + hh], z);
                            if (bias != nullptr) z = z + bv[j + hh];
                            const uint32_t cw2 = cvp[sc8 * 4 + (j + hh) / 2];
                            o[hh] = (hh ? bf16_hi(cw2) : bf16_lo(cw2)) * z;
                        }
                        pk[j / 2] = pack_bf16(o[0], o[1]);
                    }
                    if (boxed)  // 16-byte chunk sc8 of row `lane`, at position sc8 ^ (lane % 8)
                        *reinterpret_cast<uint4 *>(ybox + lane * 128 + ((sc8 ^ (lane & 7)) << 4)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    else
                        gst(reinterpret_cast<uint4 *>(y + t * (int64_t)H + h0 + c0),
                            make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    if (!single && t >= s1 - K) {  // one of the sequence's last K rows: its u to the tail
                        const int m = (int)(K - (s1 - t));
                        const uint16_t *ur = reinterpret_cast<const uint16_t *>(urow + c0 * 2);
                        uint16_t *tl = reinterpret_cast<uint16_t *>(tail);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            gst(tl + ((int64_t)i * H + h0 + c0 + j) * K + m, ur[j]);
                    }
                }
            }
            if (boxed) {  // rows past T and channels past H are not written
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_y, smem_addr(ybox), h0 + cw, (int)box_row);
                    bulk_commit();
                }
            }
            named_sync(1, kInEpiThreads);  // u_tile, taps and bias free for the next tile
        }
        if (lane == 0) bulk_wait_read<0>();  // the ring stays valid until the stores read it
        __syncwarp();
        fin_ok = all && !bad;
    }
    pipe_finish<CL>(tmem);

    // Single-sequence schedule: the CTA that ran the sequence's last row tile
    // (its last tile, so u_tile still holds it) writes the new state of the
    // tile's channels: the last K entries of [old state; u]. The cluster
    // barrier in pipe_finish ordered every read of the old state (the
    // column's first row tile, in this cluster) before these writes.
    if (single && warp >= 2 && fin_ok && fin_mt == n_mtiles - 1) {
        const int et = threadIdx.x - 64;
        const int h0 = fin_ct * kConvCh;
        const int32_t slot = gld(slots);
        const int64_t row0 = (int64_t)fin_mt * OUT - (K - 1);  // global row of tile row 0
        if (slot < 0 || slot >= n_slots) {
            if (et == 0) raise_error(SC_DEV_BAD_SLOT);
        } else {
            for (int c = et; c < kConvCh && h0 + c < H; c += kInEpiThreads) {
                bf16 *dst = pool + ((int64_t)slot * H + h0 + c) * K;
                bf16 nv[K];
#pragma unroll
                for (int m = 0; m < K; ++m) {
                    const int64_t e = T_rows + m;  // index into [old state; u_0 .. u_{T-1}]
                    nv[m] = e < K ? gld(dst + e)
                                  : *reinterpret_cast<const bf16 *>(
                                        u_tile + (e - K - row0) * kUStride + c * 2);
                }
#pragma unroll
                for (int m = 0; m < K; ++m) gst(dst + m, nv[m]);
            }
        }
    }
}

// New state of sequence i = the last K entries of [old state; u of its rows]:
// entry m is old[len + m] when len + m < K, else tail[i][h][m]. One thread per
// (sequence, 8 channels); nothing for empty sequences. A thread's 8 channels x
// K taps are 16 K contiguous bytes in the pool and in the tail, moved as
// 16-byte words. Everything that does not depend on the slot id is requested
// at once after the wait; the old state is read only for sequences shorter
// than K, the only ones whose new state keeps part of it.
template <int K>
__global__ void __launch_bounds__(256)
    k_commit_states(const int32_t *__restrict__ cu, int N, int64_t T_rows,
                    const int32_t *__restrict__ slots, const uint16_t *__restrict__ tail,
                    uint16_t *__restrict__ pool, int n_slots, int H) {
    constexpr int NQ = kCh * K * 2 / 16;  // 16-byte words in a thread's block
    const int groups = H / kCh;
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = unit < (int64_t)N * groups;
    const int i = live ? (int)(unit / groups) : 0, h = (int)(unit % groups) * kCh;
    pdl_wait();
    pdl_launch_dependents();
    int bad = 0;
    for (int j = threadIdx.x; j <= N; j += blockDim.x) {
        const int32_t c = gld(cu + j);
        if (j == 0 && c != 0) bad = 1;
        if (j == N && (int64_t)c != T_rows) bad = 1;
        if (j < N && gld(cu + j + 1) < c) bad = 1;
    }
    int64_t len = 0;
    int slot = 0;
    uint4 tq[NQ];
    if (live) {
        len = (int64_t)gld(cu + i + 1) - gld(cu + i);
        slot = gld(slots + i);
        const uint4 *tp = reinterpret_cast<const uint4 *>(tail + ((int64_t)i * H + h) * K);
#pragma unroll
        for (int q = 0; q < NQ; ++q) tq[q] = gld(tp + q);
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(SC_DEV_BAD_SEQLENS);
        return;
    }
    if (!live || len == 0) return;
    if (slot < 0 || slot >= n_slots) {
        if (h == 0) raise_error(SC_DEV_BAD_SLOT);
        return;
    }
    uint4 *sp = reinterpret_cast<uint4 *>(pool + ((int64_t)slot * H + h) * K);
    if (len >= K) {  // the new state is the sequence's last K values of u
#pragma unroll
        for (int q = 0; q < NQ; ++q) gst(sp + q, tq[q]);
        return;
    }
    uint4 oq[NQ], nq[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) oq[q] = gld(sp + q);
    const uint16_t *o = reinterpret_cast<const uint16_t *>(oq);
    const uint16_t *tl = reinterpret_cast<const uint16_t *>(tq);
    uint16_t *nw = reinterpret_cast<uint16_t *>(nq);
#pragma unroll
    for (int c = 0; c < kCh; ++c)
#pragma unroll
        for (int m = 0; m < K; ++m) {
            uint16_t v = tl[c * K + m];
#pragma unroll
            for (int e = 0; e < K; ++e)  // old entry e = len + m, if it exists
                if (len + m == e) v = o[c * K + e];
            nw[c * K + m] = v;
        }
#pragma unroll
    for (int q = 0; q < NQ; ++q) gst(sp + q, nq[q]);
}

// ------------------------------------------------------------ fused in_proj + decode
//
// One token per sequence (serving decode): row i of the hidden state is
// sequence i, its conv history is the K - 1 newest values of its slot, and
// its new state is [history; u]. A CTA computes the B | C | x product block
// of kDecCh channels for 128 sequences with one N = 3 kDecCh MMA per 16-deep
// K step. With w_in seen as [3][H][D] (a 3-D tensor map), the B, C and x rows
// of the tile's channels come with one copy per stage, so TMEM columns hold
// [B | C | x]. A stage holds kDecKB such K blocks, so the MMA lane waits and
// commits once per 4 kDecKB MMAs. Two accumulator buffers let a CTA's next
// tile's MMAs overlap this tile's epilogue. Narrow tiles put every SM to work at a serving batch
// (256 sequences, H = 2048, 32 channels: 128 tiles). Each MMA carries a
// fixed cost, so single CTAs, each issuing its own MMAs, beat CTA pairs
// (one MMA stream per two SMs) here; pairs (M = 256, each CTA staging its
// half of the channels) remain a build knob.
//
// Epilogue thread = (sequence, kDecCh / 2 channels): the slot id, the state
// block and the taps are loaded while the MMAs run; then u = round(B x),
// z = sum_k w_k window_k (+ bias), y = round(C z), and the new state block is
// written back. A (sequence, channel) pair belongs to exactly one thread of
// one tile, so the slot is read and written by the same thread: no commit
// pass is needed. The arithmetic and its order are those of k_decode, so the
// results are shortconv_decode's on the bf16 projection.
#ifndef SC_DECPROJ_CH
#define SC_DECPROJ_CH 32  // channels per tile: 32 or 64
#endif
#ifndef SC_DECPROJ_CL
#define SC_DECPROJ_CL 1  // 1: single CTAs issue their own MMAs (M = 128); 2: CTA pairs (M = 256)
#endif
constexpr int kDecCL = SC_DECPROJ_CL;
static_assert(kDecCL == 1 || kDecCL == 2, "single CTAs or pairs");
constexpr int kDecCh = SC_DECPROJ_CH;
static_assert(kDecCh == 32 || kDecCh == 64, "32 or 64 channels per decode tile");
constexpr int kDecN = 3 * kDecCh;                   // B | C | x per staged channel group
constexpr int kDecHalf = kDecCh / 2;
constexpr int kDecBoxCh = kDecCh / kDecCL;          // channels a CTA stages
constexpr int kDecBufStride = kDecN <= 128 ? 128 : 256;  // TMEM columns between buffers
constexpr int kDecBufs = 2;
#ifndef SC_DECPROJ_KB
#define SC_DECPROJ_KB 2  // 64-deep K blocks per stage (each MMA lane wait covers this many)
#endif
constexpr int kDecKB = SC_DECPROJ_KB;
static_assert(kDecKB == 1 || kDecKB == 2 || kDecKB == 4, "1, 2 or 4 K blocks per stage");
constexpr uint32_t kDecBSub = 3 * kDecBoxCh * kPBK * 2;               // B, C, x rows of a block
constexpr uint32_t kDecStage = kDecKB * (kPABytes + kDecBSub);      // [A blocks][B blocks]
#ifndef SC_DECPROJ_STAGES
#define SC_DECPROJ_STAGES ((232448 - 2048) / (int)kDecStage < 8 ? (232448 - 2048) / (int)kDecStage : 8)
#endif
constexpr int kDecStages = SC_DECPROJ_STAGES;
constexpr int kDecEpiWarps = 8;                     // two per TMEM lane quarter
constexpr int kDecEpiThreads = 32 * kDecEpiWarps;
constexpr int kDecThreads = 64 + kDecEpiThreads;
constexpr int kDecChPerThread = kDecHalf;           // 16 or 32
static_assert(kDecStages <= kMaxStages, "too many stages");
static_assert(kDecStage % 1024 == 0, "stages stay 1024-byte aligned");
constexpr size_t dec_smem_bytes() { return 1024 + (size_t)kDecStages * kDecStage + sizeof(PipeState); }
static_assert(dec_smem_bytes() <= 232448, "stage ring larger than a CTA's shared memory");

template <int K>
__global__ void __launch_bounds__(kDecThreads, 1)
    k_in_proj_decode(const __grid_constant__ CUtensorMap map_h,
                     const __grid_constant__ CUtensorMap map_w3, int N, int D, int H,
                     const bf16 *__restrict__ w, const bf16 *__restrict__ bias,
                     const int32_t *__restrict__ slots, bf16 *__restrict__ pool, int n_slots,
                     bf16 *__restrict__ y, int n_ctiles, int n_mtiles) {
    constexpr int CL = kDecCL;
    constexpr int CPT = kDecChPerThread;
    constexpr int NL = CPT / 16;          // 16-column TMEM reads per part
    constexpr int SQ = CPT * K * 2 / 16;  // 16-byte words of a thread's state block
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align1024(smem_raw);
    PipeState *ps = reinterpret_cast<PipeState *>(base + (size_t)kDecStages * kDecStage);
    const uint32_t stages = smem_addr(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / kPBK;                        // 64-deep K blocks
    const int ns = (nk + kDecKB - 1) / kDecKB;      // stages per tile
    const uint32_t tmem = pipe_start<CL>(ps, &map_h, &map_w3, kDecEpiWarps);
    const TileWalk tw = tile_walk<CL>(n_mtiles, n_ctiles);

    if (warp == 0) {
        // Per K block one A box and one [3 sections][kDecBoxCh channels][64 K]
        // box; a stage holds kDecKB blocks (fewer in the last stage when nk is odd).
        if (lane == 0) {
            const bool leader = tw.rank == 0;
            uint32_t g = 0;
            bool ok = true;
            for (int grp = tw.first; grp < tw.n_groups && ok; grp += tw.step) {
                int mt, ct;
                tw.at(grp, n_ctiles, mt, ct);
                const int a_row = mt * kPBM, ch = ct * kDecCh + kDecBoxCh * tw.rank;
                for (int si = 0; si < ns; ++si, ++g) {
                    const uint32_t s = g % kDecStages;
                    if (g >= kDecStages &&
                        !mbar_wait_bounded(&ps->empty[s], (g / kDecStages - 1) & 1u)) {
                        raise_error(SC_DEV_TIMEOUT);
                        ps->abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t st = stages + s * kDecStage;
                    const int nb = min(kDecKB, nk - si * kDecKB);  // K blocks in this stage
                    const uint32_t bytes = (uint32_t)nb * (kPABytes + kDecBSub);
                    if constexpr (CL == 1) {
                        mbar_arrive_expect_tx(&ps->full[s], bytes);
                        for (int b = 0; b < nb; ++b) {
                            const int kx = (si * kDecKB + b) * kPBK;
                            tma_load_2d(st + b * kPABytes, &map_h, &ps->full[s], kx, a_row);
                            tma_load_3d(st + kDecKB * kPABytes + b * kDecBSub, &map_w3,
                                        &ps->full[s], kx, ch, 0);
                        }
                    } else {
                        const uint32_t bar = cluster_map(smem_addr(&ps->full[s]), 0);
                        if (leader) mbar_arrive_expect_tx(&ps->full[s], 2 * bytes);
                        for (int b = 0; b < nb; ++b) {
                            const int kx = (si * kDecKB + b) * kPBK;
                            tma_load_2d_pair(st + b * kPABytes, &map_h, bar, kx, a_row);
                            tma_load_3d_pair(st + kDecKB * kPABytes + b * kDecBSub, &map_w3, bar,
                                             kx, ch, 0);
                        }
                    }
                }
            }
            if (CL == 1 || leader)
                for (uint32_t c = g > kDecStages ? g - kDecStages : 0; c < g; ++c)
                    mbar_wait_bounded(&ps->full[c % kDecStages], (c / kDecStages) & 1u);
            if (ok)
                for (uint32_t c = g > kDecStages ? g - kDecStages : 0; c < g; ++c)
                    mbar_wait_bounded(&ps->empty[c % kDecStages], (c / kDecStages) & 1u);
        }
    } else if (warp == 1) {
        // One lane of the (leader) CTA: per stage, per K block, 4 MMAs of N = kDecN
        // into accumulator buffer it % 2 (as mma_tiles, with kDecKB blocks a stage).
        if (lane == 0 && tw.rank == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kPBM * CL, kDecN);
            uint32_t g = 0;
            int it = 0;
            bool ok = true;
            for (int grp = tw.first; grp < tw.n_groups && ok; grp += tw.step, ++it) {
                const int b = it % kDecBufs, use = it / kDecBufs;
                if (use >= 1 && !mbar_wait_bounded(&ps->tempty[b], (uint32_t)(use - 1) & 1u)) {
                    raise_error(SC_DEV_TIMEOUT);
                    ps->abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)b * (uint32_t)kDecBufStride;
                for (int si = 0; si < ns; ++si, ++g) {
                    const uint32_t s = g % kDecStages;
                    if (!mbar_wait_bounded(&ps->full[s], (g / kDecStages) & 1u)) {
                        raise_error(SC_DEV_TIMEOUT);
                        ps->abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = stages + s * kDecStage;
                    const int nb = min(kDecKB, nk - si * kDecKB);
                    for (int kb = 0; kb < nb; ++kb) {
                        const uint64_t da = sdesc_k128(st + kb * kPABytes);
                        const uint64_t db = sdesc_k128(st + kDecKB * kPABytes + kb * kDecBSub);
#pragma unroll
                        for (int j = 0; j < kPBK / 16; ++j) {
                            const uint32_t acc = (si | kb | j) != 0;
                            if constexpr (CL == 1)
                                mma_bf16(d, da + 2 * j, db + 2 * j, idesc, acc);
                            else
                                mma_bf16_pair(d, da + 2 * j, db + 2 * j, idesc, acc);
                        }
                    }
                    if constexpr (CL == 1)
                        mma_commit(&ps->empty[s]);
                    else
                        mma_commit_pair(&ps->empty[s], 3);
                }
                if (ok) {
                    if constexpr (CL == 1)
                        mma_commit(&ps->tfull[b]);
                    else
                        mma_commit_pair(&ps->tfull[b], 3);
                }
            }
            if constexpr (CL == 1)
                mma_commit(&ps->mma_done);
            else
                mma_commit_pair(&ps->mma_done, 1);
            mbar_wait_bounded(&ps->mma_done, 0);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;                          // TMEM lane quarter
        const int r = q * 32 + lane;                     // tile row = TMEM lane
        const int half = (warp - 2) >> 2;                // this thread's half of the channels
        const int cpart = half * CPT;                    // its first channel in the tile
        // TMEM columns of its B, C and x values. Pairs: [B | C | x] of each
        // CTA's half of the channels in turn; single CTAs: [B | C | x] of all.
        const uint32_t col_b = CL == 2 ? (uint32_t)(3 * cpart) : (uint32_t)cpart;
        const uint32_t col_c = col_b + kDecBoxCh;
        const uint32_t col_x = col_b + 2 * kDecBoxCh;
        int it = 0;
        for (int grp = tw.first; grp < tw.n_groups; grp += tw.step, ++it) {
            int mt, ct;
            tw.at(grp, n_ctiles, mt, ct);
            const int h = ct * kDecCh + cpart;           // first channel of the thread
            const int64_t i = (int64_t)mt * kPBM + r;    // sequence
            // Everything that does not depend on the product, while the MMAs run.
            bool live = i < N;
            int slot = 0;
            uint4 sq[SQ];
            uint32_t wq[CPT * K / 2], bq[CPT / 2];
            if (live) {
                slot = gld(slots + i);
                if (slot < 0 || slot >= n_slots) {
                    if (h == 0) raise_error(SC_DEV_BAD_SLOT);
                    live = false;
                }
            }
            if (live) {
                const uint4 *sp = reinterpret_cast<const uint4 *>(pool + ((int64_t)slot * H + h) * K);
#pragma unroll
                for (int e = 0; e < SQ; ++e) sq[e] = gld(sp + e);
                const uint32_t *wp = reinterpret_cast<const uint32_t *>(w + (int64_t)h * K);
#pragma unroll
                for (int e = 0; e < CPT * K / 2; ++e) wq[e] = gld(wp + e);
                if (bias != nullptr) {
                    const uint32_t *bp = reinterpret_cast<const uint32_t *>(bias + h);
#pragma unroll
                    for (int e = 0; e < CPT / 2; ++e) bq[e] = gld(bp + e);
                }
            }
            if (!epi_acquire<kDecBufs>(ps, it, kDecEpiThreads)) break;
            const uint32_t trow = tmem + (uint32_t)(it % kDecBufs) * (uint32_t)kDecBufStride +
                                  ((uint32_t)(q * 32) << 16);
            uint32_t rb[NL][16], rc[NL][16], rx[NL][16];
            __syncwarp();  // tcgen05.ld is warp-collective
#pragma unroll
            for (int l = 0; l < NL; ++l) {
                tmem_ld16_nowait(trow + col_b + 16 * l, rb[l]);
                tmem_ld16_nowait(trow + col_c + 16 * l, rc[l]);
                tmem_ld16_nowait(trow + col_x + 16 * l, rx[l]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int l = 0; l < NL; ++l) {
                tmem_regs_ready(rb[l]);
                tmem_regs_ready(rc[l]);
                tmem_regs_ready(rx[l]);
            }
            epi_release<CL, kDecBufs>(ps, it, tw.rank);  // the accumulator buffer is read
            if (!live) continue;
            uint32_t sw[4 * SQ];  // the state block as words: element e in half e % 2 of word e / 2
#pragma unroll
            for (int e = 0; e < SQ; ++e) {
                sw[4 * e] = sq[e].x;
                sw[4 * e + 1] = sq[e].y;
                sw[4 * e + 2] = sq[e].z;
                sw[4 * e + 3] = sq[e].w;
            }
            auto elem = [](const uint32_t *wd, int e) {
                return (e & 1) ? bf16_hi(wd[e >> 1]) : bf16_lo(wd[e >> 1]);
            };
            uint32_t yw[CPT / 2];
            float ns[CPT * K];  // the new state block, bf16 values
#pragma unroll
            for (int c = 0; c < CPT; c += 2) {
                const int l = c / 16, j = c % 16;
                // B, x and C rounded to bf16 (the values a separate in_proj stores);
                // u = round(B x), the exact product rounded once
                const uint32_t bx =
                    bf2_mul(pack_bf16(__uint_as_float(rb[l][j]), __uint_as_float(rb[l][j + 1])),
                            pack_bf16(__uint_as_float(rx[l][j]), __uint_as_float(rx[l][j + 1])));
                const uint32_t cc =
                    pack_bf16(__uint_as_float(rc[l][j]), __uint_as_float(rc[l][j + 1]));
                float o[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ch = c + hh;
                    float win[K], wk[K];
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        win[k] = elem(sw, ch * K + k);
                        wk[k] = elem(wq, ch * K + k);
                    }
                    const float u = hh ? bf16_hi(bx) : bf16_lo(bx);
                    float z = slide_dot<K>(win, wk, u);
                    if (bias != nullptr) z = z + elem(bq, ch);
                    o[hh] = (hh ? bf16_hi(cc) : bf16_lo(cc)) * z;
#pragma unroll
                    for (int k = 0; k < K; ++k) ns[ch * K + k] = win[k];
                }
                yw[c / 2] = pack_bf16(o[0], o[1]);
            }
            uint4 *yp = reinterpret_cast<uint4 *>(y + i * (int64_t)H + h);
#pragma unroll
            for (int e = 0; e < CPT / 8; ++e)
                gst(yp + e, make_uint4(yw[4 * e], yw[4 * e + 1], yw[4 * e + 2], yw[4 * e + 3]));
            uint32_t nw[4 * SQ];  // exact: every value is a bf16 already
#pragma unroll
            for (int m = 0; m < 4 * SQ; ++m)
                nw[m] = (__float_as_uint(ns[2 * m]) >> 16) | (__float_as_uint(ns[2 * m + 1]) & 0xFFFF0000u);
            uint4 *sp = reinterpret_cast<uint4 *>(pool + ((int64_t)slot * H + h) * K);
#pragma unroll
            for (int e = 0; e < SQ; ++e)
                gst(sp + e, make_uint4(nw[4 * e], nw[4 * e + 1], nw[4 * e + 2], nw[4 * e + 3]));
        }
    }
    pipe_finish<CL>(tmem);
}

// ------------------------------------------------------------ out_proj

template <int CL>
__global__ void __launch_bounds__(kOutThreads, 1)
    k_out_proj(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_o, int Kdim, int n_ntiles, int n_mtiles) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = align1024(smem_raw);
    unsigned char *stg_all = base + (size_t)kOutStages * kOutStage;
    PipeState *ps = reinterpret_cast<PipeState *>(stg_all + kOutStg);
    const uint32_t stages = smem_addr(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = Kdim / kPBK;
    const uint32_t tmem = pipe_start<CL>(ps, &map_a, &map_b, 4);
    const TileWalk tw = tile_walk<CL>(n_mtiles, n_ntiles);

    if (warp == 0) {
        auto out_coords = [&](int mt, int nt, int &a_row, int (&rows)[1]) {
            a_row = mt * kPBM;
            rows[0] = nt * kOutN + tw.rank * kOutBoxRows;
        };
        if (lane == 0)
            produce_tiles<kOutStages, 1, CL>(
                &map_a, &map_b, stages, kOutStage, ps, nk, tw, n_ntiles, kOutBox, out_coords);
    } else if (warp == 1) {
        if (lane == 0 && tw.rank == 0)
            mma_tiles<kOutStages, kOutN, 0, CL, kOutBufs>(tmem, stages, kOutStage, ps, nk, tw);
        __syncwarp();
    } else {
        // Warp q drains TMEM lanes 32q .. 32q + 31 (tile rows) in boxes of 64
        // columns: rounded to bf16 into a staging box and stored by lane 0
        // with a TMA copy (rows past the end are not written). Boxes alternate
        // between the warp's two staging boxes, except in the CTA's last tile:
        // its MMAs have consumed every stage and no load follows, so the
        // stage ring holds all of its boxes and no store waits for another.
        if (lane == 0) tma_prefetch_map(&map_o);
        const int q = warp & 3;
        unsigned char *stg = stg_all + (size_t)q * 2 * kOutStgBox;
        unsigned char *ring = base + (size_t)q * kOutBoxes * kOutStgBox;
        uint32_t nbox = 0;  // staging boxes this warp has filled
        int it = 0;
        for (int grp = tw.first; grp < tw.n_groups; grp += tw.step, ++it) {
            int mt, nt;
            tw.at(grp, n_ntiles, mt, nt);
            const int row0 = mt * kPBM + q * 32;
            const int col0 = nt * kOutN;
            const bool last = grp + tw.step >= tw.n_groups;
            if (!epi_acquire<kOutBufs>(ps, it, 128)) break;
            const uint32_t trow =
                tmem + (uint32_t)(it % kOutBufs) * 256u + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int bx = 0; bx < kOutBoxes; ++bx) {
                uint32_t r[4][16];
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) tmem_ld16_nowait(trow + bx * kPBK + i * 16, r[i]);
                unsigned char *buf;
                if (last) {
                    buf = ring + (size_t)bx * kOutStgBox;
                } else {
                    buf = stg + (nbox++ & 1u) * kOutStgBox;
                    if (lane == 0) bulk_wait_read<1>();  // the store that last read buf is done
                }
                __syncwarp();
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 4; ++i) tmem_regs_ready(r[i]);
                // Row `lane` of the box: 16-byte chunk j (columns 8j .. 8j + 7)
                // goes to chunk position j ^ (row % 8) of the row's 128 bytes.
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *v = &r[j >> 1][(j & 1) * 8];
                    uint4 pk;
                    pk.x = pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1]));
                    pk.y = pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3]));
                    pk.z = pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5]));
                    pk.w = pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7]));
                    *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = pk;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_o, smem_addr(buf), col0 + bx * kPBK, row0);
                    bulk_commit();
                }
            }
            epi_release<CL, kOutBufs>(ps, it, tw.rank);
        }
        if (lane == 0) bulk_wait_read<0>();  // staging stays valid until every store has read it
        __syncwarp();
    }
    pipe_finish<CL>(tmem);
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

// A row-major bf16 matrix [outer, inner] copied in {64, box_rows} boxes with
// the 128-byte swizzle; a load reads rows past the end (or before row 0) as
// zeros, a store leaves them unwritten.
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

// w_in [3H, D] seen as [3][H][D]: a box covers 64 K values of `box_rows`
// channels in each of the three sections (B, C, x), written to shared memory
// section after section (3 box_rows rows of 128 bytes, 128-byte swizzle).
static cudaError_t map_3d_sections(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t H,
                                   uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {inner, H, 3};
    const cuuint64_t strides[2] = {inner * 2, H * inner * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kPBK, box_rows, 3};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
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

// How many clusters of kPCluster CTAs of `kern` fit on the device at once
// (the persistent grid), cached per device.
template <typename F>
static cudaError_t max_clusters(F kern, size_t smem, int threads, int sm_count,
                                std::atomic<int> (&cache)[64],
                                int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cache[dev].load() > 0) {
        *out = cache[dev].load();
        return cudaSuccess;
    }
    int n = sm_count / kPCluster;
    if (kPCluster > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(kPCluster * (sm_count / kPCluster)));
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kPCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, (const void *)kern, &cfg);
        if (e != cudaSuccess) return e;
    }
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) cache[dev].store(n);
    *out = n;
    return cudaSuccess;
}

size_t in_proj_workspace_bytes(int H, int K, int N) { return (size_t)N * H * K * 2; }

template <int K>
static cudaError_t in_proj_inst(const CUtensorMap &mh, const CUtensorMap &mw, const CUtensorMap &my,
                                int64_t T, int D,
                                int H, const void *w, const void *bias, const int32_t *cu, int N,
                                const int32_t *slots, void *pool, int n_slots, void *y,
                                void *tail, int sm_count, cudaStream_t stream) {
    constexpr int OUT = kPBM - (K - 1);
    cudaError_t e;
    bool single = false;  // one sequence: the fused kernel writes its new state itself
    if (T > 0) {
        auto kern = k_in_proj_conv<K, kPCluster>;
        static std::atomic<unsigned long long> done{0};
        e = smem_opt_in(kern, conv_smem_bytes(), done);
        if (e != cudaSuccess) return e;
        static std::atomic<int> cache[64];
        int clusters = 0;
        e = max_clusters(kern, conv_smem_bytes(), kInThreads, sm_count, cache, &clusters);
        if (e != cudaSuccess) return e;
        const int n_ctiles = (H + kConvCh - 1) / kConvCh;  // the last may be half full
        const int64_t n_mtiles = (T + OUT - 1) / OUT;
        const int64_t pairs = (n_mtiles + kPCluster - 1) / kPCluster;
        const int64_t groups = pairs * n_ctiles;
        const int grid = kPCluster * (int)(groups < clusters ? groups : clusters);  // persistent
        // The single-sequence walk needs every column's first and last pair in
        // one cluster, the last one being that cluster's last tile.
        single = N == 1 && n_ctiles <= clusters &&
                 (pairs == 1 || groups >= (int64_t)clusters + n_ctiles);
        e = launch_pdl_cluster(kern, dim3((unsigned)grid), dim3(kInThreads), conv_smem_bytes(),
                               stream, kPCluster, mh, mw, my, T, D, H, (const bf16 *)w,
                               (const bf16 *)bias, cu, N, slots, (bf16 *)pool, n_slots,
                               (bf16 *)y, (bf16 *)tail, n_ctiles, (int)n_mtiles, single ? 1 : 0);
        if (e != cudaSuccess) return e;
    }
    if (single) return cudaSuccess;  // no commit pass
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
    CUtensorMap mh, mw, my;
    if (T > 0) {
        cudaError_t e = map_2d(&mh, hidden, (uint64_t)D, (uint64_t)T, kPBM);
        if (e != cudaSuccess) return e;
        e = map_2d(&mw, w_in, (uint64_t)D, (uint64_t)3 * H, kConvBoxRows);
        if (e != cudaSuccess) return e;
        e = map_2d(&my, y, (uint64_t)H, (uint64_t)T, 32);
        if (e != cudaSuccess) return e;
    }
    switch (K) {
        case 1: return in_proj_inst<1>(mh, mw, my, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        case 2: return in_proj_inst<2>(mh, mw, my, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        case 3: return in_proj_inst<3>(mh, mw, my, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
        default: return in_proj_inst<4>(mh, mw, my, T, D, H, w, bias, cu, N, slots, pool, n_slots, y, workspace, sm_count, stream);
    }
}

template <int K>
static cudaError_t in_proj_decode_inst(const CUtensorMap &mh, const CUtensorMap &mw3, int N,
                                       int D,
                                       int H, const void *w, const void *bias,
                                       const int32_t *slots, void *pool, int n_slots, void *y,
                                       int sm_count, cudaStream_t stream) {
    auto kern = k_in_proj_decode<K>;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = smem_opt_in(kern, dec_smem_bytes(), done);
    if (e != cudaSuccess) return e;
    int clusters = sm_count;  // single CTAs: one per SM (the stage ring fills its shared memory)
    if (kDecCL == 2) {
        static std::atomic<int> cache[64];
        e = max_clusters(kern, dec_smem_bytes(), kDecThreads, sm_count, cache, &clusters);
        if (e != cudaSuccess) return e;
    }
    const int n_ctiles = H / kDecCh;
    const int n_mtiles = (N + kPBM - 1) / kPBM;
    const int64_t groups = (int64_t)(n_mtiles + kDecCL - 1) / kDecCL * n_ctiles;
    const int grid = kDecCL * (int)(groups < clusters ? groups : clusters);  // persistent
    return launch_pdl_cluster(kern, dim3((unsigned)grid), dim3(kDecThreads), dec_smem_bytes(),
                              stream, (unsigned)kDecCL, mh, mw3, N, D, H, (const bf16 *)w,
                              (const bf16 *)bias,
                              slots, (bf16 *)pool, n_slots, (bf16 *)y, n_ctiles, n_mtiles);
}

cudaError_t launch_in_proj_decode(int D, int H, int K, const void *hidden, int N,
                                  const void *w_in, const void *w, const void *bias,
                                  const int32_t *slots, void *pool, int n_slots, void *y,
                                  int sm_count, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    CUtensorMap mh;
    cudaError_t e = map_2d(&mh, hidden, (uint64_t)D, (uint64_t)N, kPBM);
    if (e != cudaSuccess) return e;
    CUtensorMap mw3;  // w_in as [3 sections][H channels][D]: boxes of all three sections
    e = map_3d_sections(&mw3, w_in, (uint64_t)D, (uint64_t)H, (uint32_t)kDecBoxCh);
    if (e != cudaSuccess) return e;
    switch (K) {
        case 1: return in_proj_decode_inst<1>(mh, mw3, N, D, H, w, bias, slots, pool, n_slots, y, sm_count, stream);
        case 2: return in_proj_decode_inst<2>(mh, mw3, N, D, H, w, bias, slots, pool, n_slots, y, sm_count, stream);
        case 3: return in_proj_decode_inst<3>(mh, mw3, N, D, H, w, bias, slots, pool, n_slots, y, sm_count, stream);
        default: return in_proj_decode_inst<4>(mh, mw3, N, D, H, w, bias, slots, pool, n_slots, y, sm_count, stream);
    }
}

cudaError_t launch_out_proj(int H, int D, const void *y, int64_t T, const void *w_out, void *out,
                            int sm_count, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    CUtensorMap ma, mb, mo;
    cudaError_t e = map_2d(&ma, y, (uint64_t)H, (uint64_t)T, kPBM);
    if (e != cudaSuccess) return e;
    e = map_2d(&mb, w_out, (uint64_t)H, (uint64_t)D, kOutBoxRows);
    if (e != cudaSuccess) return e;
    e = map_2d(&mo, out, (uint64_t)D, (uint64_t)T, 32);
    if (e != cudaSuccess) return e;
    auto kern = k_out_proj<kPCluster>;
    static std::atomic<unsigned long long> done{0};
    e = smem_opt_in(kern, out_smem_bytes(), done);
    if (e != cudaSuccess) return e;
    static std::atomic<int> cache[64];
    int clusters = 0;
    e = max_clusters(kern, out_smem_bytes(), kOutThreads, sm_count, cache, &clusters);
    if (e != cudaSuccess) return e;
    const int n_ntiles = D / kOutN;
    const int64_t n_mtiles = (T + kPBM - 1) / kPBM;
    const int64_t groups = (n_mtiles + kPCluster - 1) / kPCluster * n_ntiles;
    const int grid = kPCluster * (int)(groups < clusters ? groups : clusters);  // persistent
    return launch_pdl_cluster(kern, dim3((unsigned)grid), dim3(kOutThreads), out_smem_bytes(),
                              stream, kPCluster, ma, mb, mo, H, n_ntiles, (int)n_mtiles);
}

cudaError_t take_error_proj(cudaStream_t stream, unsigned int *code) {
    return take_error_here(stream, code);
}

#ifdef SC_BOUNDS_CHECK
cudaError_t bounds_install_proj(const BoundsRegion *r, int n, cudaStream_t stream) {
    return bounds_install_here(r, n, stream);
}
cudaError_t bounds_take_proj(cudaStream_t stream, unsigned long long *addr) {
    return bounds_take_first_bad_here(stream, addr);
}
#endif

}  // namespace sc
