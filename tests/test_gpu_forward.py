"""GPU forward path (prefill, decode, verify, rollback) against the CPU oracle.

Every call goes through the C ABI (via the ctypes binding) on seeded inputs
shared with the oracle: conv states and verify windows must match bit for
bit, outputs within the tolerances in gpu_util.
"""
import numpy as np
import pytest
import torch

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from fixtures import tiny_fp32_golden, worked_example
from gpu_util import assert_bits, assert_close, dev, host

pytestmark = pytest.mark.gpu

TILES = [0, 4, 8, 16, 32]  # 0: the TMA-streamed kernel; others: register-tiled rows per thread


def run_prefill(p, tile=0):
    pool = dev(p.pool, p.dtype)
    y = sc.prefill(dev(p.bcx, p.dtype), dev(p.w, p.dtype), dev(p.cu_seqlens, "i32"),
                   dev(p.slot_ids, "i32"), pool, rows_per_thread=tile)
    torch.cuda.synchronize()
    return host(y), host(pool)


def oracle_prefill(p):
    pool = p.pool.copy()
    st, y = oracle.prefill(p.dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, pool)
    assert st == oracle.OK
    return y, pool


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_example(dtype):
    ex = worked_example(dtype)
    pool = dev(ex["state"][None], dtype)
    y = sc.prefill(dev(ex["bcx"], dtype), dev(ex["w"], dtype), dev(np.array([0, 4]), "i32"),
                   dev(np.array([0]), "i32"), pool)
    assert_bits(host(y), ex["y"], "y")
    assert_bits(host(pool)[0], ex["final_state"], "state")


def test_tiny_fp32_config_against_golden_and_oracle():
    """One fp32 sequence, H=64, K=3, T=16 from zero state, then 4 decode tokens."""
    g = tiny_fp32_golden()
    pool = torch.zeros((1, g["H"], g["K"]), dtype=torch.float32, device="cuda")
    w = dev(g["w"], "f32")
    y = sc.prefill(dev(g["bcx"], "f32"), w, dev(np.array([0, g["T"]]), "i32"),
                   dev(np.array([0]), "i32"), pool)
    assert_close("f32", host(y), g["y_prefill"], "y prefill")
    assert_bits(host(pool)[0], g["state_after_prefill"], "state after prefill")
    slot = dev(np.array([0]), "i32")
    for s in range(g["steps"]):
        yd = sc.decode(dev(g["decode_bcx"][s], "f32"), w, slot, pool)
        assert_close("f32", host(yd)[0], g["y_decode"][s], f"y decode {s}")
    assert_bits(host(pool)[0], g["state_after_decode"], "state after decode")
    assert sc.get_error() == 0


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_sequence_ragged(dtype, tile, K):
    p = wl.single_prefill(T=301, H=256, K=K, seed=10 + K, dtype=dtype)
    p.pool = wl.normal(np.random.default_rng(K), (1, 256, K), 1.0, dtype)  # continued prefill
    y, pool = run_prefill(p, tile)
    y_ref, pool_ref = oracle_prefill(p)
    assert_close(dtype, y, y_ref, "y")
    assert_bits(pool, pool_ref, "state")


@pytest.mark.parametrize("T", [1, 2, 3, 5])
def test_sequences_shorter_than_the_window(T):
    p = wl.single_prefill(T=T, H=64, K=4, seed=20 + T)
    p.pool = wl.normal(np.random.default_rng(T), (1, 64, 4), 1.0, "bf16")
    y_ref, pool_ref = oracle_prefill(p)
    for tile in (0, 4):
        y, pool = run_prefill(p, tile)
        assert_close("bf16", y, y_ref, "y")
        assert_bits(pool, pool_ref, "state")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("K", [2, 3, 4])
def test_varlen_with_empty_and_tiny_sequences(tile, K):
    lengths = [0, 1, 2, 3, 5, 64, 100, 7, 0, 33, 4, 1, 0, 31, 32, 9]
    p = wl.varlen_prefill(H=128, K=K, n_slots=40, seed=30 + K, lengths=lengths)
    y, pool = run_prefill(p, tile)
    y_ref, pool_ref = oracle_prefill(p)
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool (named and untouched slots)")


def test_tiles_give_identical_bits():
    p = wl.varlen_prefill(n_seqs=9, lo=1, hi=300, H=256, K=3, n_slots=16, seed=40)
    outs = [run_prefill(p, t) for t in TILES]
    for y, pool in outs[1:]:
        assert_bits(y, outs[0][0], "y across tiles")
        assert_bits(pool, outs[0][1], "pool across tiles")


@pytest.mark.parametrize("H", [2560, 4096])
def test_channel_slices_wider_than_one_cta(H):
    p = wl.varlen_prefill(n_seqs=5, lo=1, hi=90, H=H, K=3, n_slots=7, seed=41)
    outs = [run_prefill(p, t) for t in (0, 8)]
    y_ref, pool_ref = oracle_prefill(p)
    for y, pool in outs:
        assert_close("bf16", y, y_ref, "y")
        assert_bits(pool, pool_ref, "pool")


def test_more_sequences_than_staged_in_shared_memory():
    rng = np.random.default_rng(42)
    lengths = rng.integers(0, 4, size=2100)
    p = wl.varlen_prefill(H=64, K=3, n_slots=2200, seed=42, lengths=lengths)
    y_ref, pool_ref = oracle_prefill(p)
    for t in (0, 4):
        y, pool = run_prefill(p, t)
        assert_close("bf16", y, y_ref, "y")
        assert_bits(pool, pool_ref, "pool")


@pytest.mark.parametrize("T", [1, 7, 9, 17, 1217])
def test_stream_kernel_row_split_edges(T):
    """Few rows per CTA: halo and owner extensions cross many CTA boundaries."""
    p = wl.varlen_prefill(H=256, K=4, n_slots=T + 2, seed=43 + T,
                          lengths=np.diff(np.unique(np.r_[0, np.random.default_rng(T).integers(
                              0, T, size=max(1, T // 3)), T])))
    y_ref, pool_ref = oracle_prefill(p)
    y, pool = run_prefill(p, 0)
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool")


def test_prefill_T4096_H2048_full_size():
    """LFM2-1.2B-shaped single-sequence prefill (T=4096, H=2048, K=3), automatic tile."""
    p = wl.single_prefill()
    y, pool = run_prefill(p, 0)
    y_ref, pool_ref = oracle_prefill(p)
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "state")


def test_packed_varlen_16_sequences_full_size():
    """16 sequences, lengths U{64..2048}, 1024-slot pool, half continued from N(0,1) states."""
    p = wl.varlen_prefill()
    y, pool = run_prefill(p, 0)
    y_ref, pool_ref = oracle_prefill(p)
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool")


def test_chunked_prefill_and_decode_equal_full_prefill_on_gpu():
    p = wl.single_prefill(T=200, H=256, K=3, seed=50)
    y_full, pool_full = run_prefill(p, 8)
    bcx = dev(p.bcx, "bf16")
    w = dev(p.w, "bf16")
    pool = dev(p.pool, "bf16")
    slot = dev(np.array([0]), "i32")
    ys = []
    for a, b in [(0, 1), (1, 2), (2, 70), (70, 71), (71, 150)]:
        ys.append(sc.prefill(bcx[a:b].contiguous(), w, dev(np.array([0, b - a]), "i32"), slot,
                             pool))
    for t in range(150, 200):
        ys.append(sc.decode(bcx[t:t + 1].contiguous(), w, slot, pool))
    assert_bits(host(torch.cat(ys)), y_full, "y")
    assert_bits(host(pool), pool_full, "state")


# ------------------------------------------------------------------- decode

@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(dtype, K):
    s = wl.decode_serving(layers=1, steps=3, batch=37, H=64, K=K, n_slots=50, seed=60 + K,
                          dtype=dtype)
    pool = dev(s.pools[0], dtype)
    ref = s.pools[0].copy()
    w = dev(s.w[0], dtype)
    slots = dev(s.slot_ids, "i32")
    for step in range(3):
        y = sc.decode(dev(s.bcx[0, step], dtype), w, slots, pool)
        st, y_ref = oracle.decode(dtype, s.bcx[0, step], s.w[0], s.slot_ids, ref)
        assert st == oracle.OK
        assert_close(dtype, host(y), y_ref, f"y step {step}")
    assert_bits(host(pool), ref, "pool")


def test_decode_serving_256_sequences_two_layers():
    """bs=256 decode, H=2048, 1024-slot pools, 2 layers x 8 steps of the serving workload."""
    s = wl.decode_serving(layers=2, steps=8)
    for layer in range(2):
        pool = dev(s.pools[layer], "bf16")
        ref = s.pools[layer].copy()
        w = dev(s.w[layer], "bf16")
        slots = dev(s.slot_ids, "i32")
        for step in range(8):
            y = sc.decode(dev(s.bcx[layer, step], "bf16"), w, slots, pool)
            st, y_ref = oracle.decode("bf16", s.bcx[layer, step], s.w[layer], s.slot_ids, ref)
            assert st == oracle.OK
            assert_close("bf16", host(y), y_ref, f"layer {layer} step {step}")
        assert_bits(host(pool), ref, f"pool layer {layer}")


@pytest.mark.parametrize("op", ["decode", "verify"])
def test_slot_ids_rewritten_by_the_kernel_just_before(op):
    """Decode and verify read each slot id once before their dependency wait,
    only to prefetch that slot's state into L2. Here the
    kernel just before them in the stream, a device-side slot claim, rewrites
    the slot-id buffer they read, so that early read can see the old ids. The
    results must follow the claimed slots, and the old slots must stay as they
    were."""
    from oracle import slots as model
    rng = np.random.default_rng(31)
    n_slots, H, K, N, D = 96, 512, 3, 24, 4
    for it in range(6):
        bm = np.zeros(model.words(n_slots), np.uint32)
        for s_ in rng.choice(n_slots, size=40, replace=False):
            bm[s_ // 32] |= np.uint32(1 << (int(s_) % 32))
        pool0 = oracle.round_bf16(rng.standard_normal((n_slots, H, K)))
        w = oracle.round_bf16(rng.standard_normal((H, K)) * 0.6)
        rows = N if op == "decode" else N * D
        bcx = oracle.round_bf16(rng.standard_normal((rows, 3 * H)))
        ref_bm, ref_pool = bm.copy(), pool0.copy()
        st, claimed = model.claim(ref_bm, n_slots, N, pool=ref_pool)
        assert st == model.OK
        # the buffer first holds other valid ids: slots that the claim does not take
        old = rng.permutation(np.setdiff1d(np.arange(n_slots), claimed))[:N].astype(np.int32)
        slot_buf = dev(old, "i32")
        pool = dev(pool0, "bf16")
        d_bm = torch.from_numpy(bm.view(np.int32).copy()).cuda()
        torch.cuda.synchronize()
        sc.slots_claim(d_bm, n_slots, N, pool=pool, slots_out=slot_buf)
        if op == "decode":
            y = sc.decode(dev(bcx, "bf16"), dev(w, "bf16"), slot_buf, pool)
            st, y_ref = oracle.decode("bf16", bcx, w, claimed, ref_pool)
            assert st == oracle.OK
            assert_close("bf16", host(y), y_ref, f"y, pass {it}")
        else:
            win, y = sc.verify(dev(bcx, "bf16"), dev(w, "bf16"), slot_buf, pool, D)
            st, win_ref, y_ref = oracle.verify("bf16", bcx, w, claimed, ref_pool, D)
            assert st == oracle.OK
            assert_close("bf16", host(y), y_ref, f"y, pass {it}")
            assert_bits(host(win), win_ref, f"win, pass {it}")
        assert_bits(host(slot_buf), claimed, f"claimed ids, pass {it}")
        assert_bits(host(pool), ref_pool, f"pool, pass {it}")
        assert sc.get_error() == 0


# ----------------------------------------------------------- verify/rollback

@pytest.mark.parametrize("D", [1, 3, 4, 8, 12])
@pytest.mark.parametrize("K", [1, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_and_rollback_small(dtype, K, D):
    s = wl.verify_serving(layers=1, batch=9, D=D, H=64, K=K, n_slots=12, seed=70 + D + K,
                          dtype=dtype)
    pool = dev(s.pools[0], dtype)
    win, y = sc.verify(dev(s.bcx[0], dtype), dev(s.w[0], dtype), dev(s.slot_ids, "i32"), pool, D)
    st, win_ref, y_ref = oracle.verify(dtype, s.bcx[0], s.w[0], s.slot_ids, s.pools[0], D)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, "y")
    assert_bits(host(win), win_ref, "win")
    assert_bits(host(pool), s.pools[0], "pool untouched by verify")
    sc.rollback(win, dev(s.accepted, "i32"), dev(s.slot_ids, "i32"), pool)
    ref = s.pools[0].copy()
    assert oracle.rollback(dtype, win_ref, s.accepted, s.slot_ids, ref) == oracle.OK
    assert_bits(host(pool), ref, "pool after rollback")
    assert sc.get_error() == 0


def test_verify_64x8_full_width_then_rollback():
    """64 sequences x 8 drafts, H=2048, 1024-slot pool, accepted ~ U{0..8}."""
    s = wl.verify_serving(layers=1)
    pool = dev(s.pools[0], "bf16")
    win, y = sc.verify(dev(s.bcx[0], "bf16"), dev(s.w[0], "bf16"), dev(s.slot_ids, "i32"),
                       pool, s.D)
    st, win_ref, y_ref = oracle.verify("bf16", s.bcx[0], s.w[0], s.slot_ids, s.pools[0], s.D)
    assert st == oracle.OK
    assert_close("bf16", host(y), y_ref, "y")
    assert_bits(host(win), win_ref, "win")
    sc.rollback(win, dev(s.accepted, "i32"), dev(s.slot_ids, "i32"), pool)
    ref = s.pools[0].copy()
    assert oracle.rollback("bf16", win_ref, s.accepted, s.slot_ids, ref) == oracle.OK
    assert_bits(host(pool), ref, "pool after rollback")


def test_rollback_equals_decoding_the_accepted_prefix_on_gpu():
    s = wl.verify_serving(layers=1, batch=16, D=5, H=128, K=3, n_slots=20, seed=80)
    s.accepted = np.arange(16, dtype=np.int32) % 6
    pool_v = dev(s.pools[0], "bf16")
    w = dev(s.w[0], "bf16")
    win, _ = sc.verify(dev(s.bcx[0], "bf16"), w, dev(s.slot_ids, "i32"), pool_v, s.D)
    sc.rollback(win, dev(s.accepted, "i32"), dev(s.slot_ids, "i32"), pool_v)
    pool_d = dev(s.pools[0], "bf16")
    rows = s.bcx[0].reshape(16, s.D, -1)
    for j in range(s.D):
        take = np.nonzero(s.accepted > j)[0]
        if len(take):
            sc.decode(dev(rows[take, j], "bf16"), w, dev(s.slot_ids[take], "i32"), pool_d)
    assert_bits(host(pool_v), host(pool_d), "rollback vs decode")


def test_graph_captured_layers_match_eager_calls():
    """Decode, verify and rollback captured in one CUDA graph (dependent launches
    chained through the shared pools) give the same bits as eager calls."""
    s = wl.decode_serving(layers=3, steps=2, batch=64, H=512, K=3, n_slots=128, seed=110)
    v = wl.verify_serving(layers=3, batch=16, D=4, H=512, K=3, n_slots=128, seed=111)

    def run(graph: bool):
        pools = [dev(s.pools[l], "bf16") for l in range(3)]
        w = [dev(s.w[l], "bf16") for l in range(3)]
        slots = dev(s.slot_ids, "i32")
        vs = dev(s.slot_ids[:16], "i32")  # verify on slots the decode just wrote (distinct)
        acc = dev(v.accepted, "i32")
        bcx = [[dev(s.bcx[l, t], "bf16") for t in range(2)] for l in range(3)]
        vb = [dev(v.bcx[l], "bf16") for l in range(3)]
        ys = [torch.empty((64, 512), dtype=torch.bfloat16, device="cuda") for _ in range(6)]
        wins = [torch.empty((16, 4, 512, 3), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        yv = [torch.empty((64, 512), dtype=torch.bfloat16, device="cuda") for _ in range(3)]

        def body():
            for t in range(2):
                for l in range(3):
                    sc.decode(bcx[l][t], w[l], slots, pools[l], y=ys[3 * t + l])
            for l in range(3):
                sc.verify(vb[l], w[l], vs, pools[l], 4, win=wins[l], y=yv[l])
                sc.rollback(wins[l], acc, vs, pools[l])

        if graph:
            side = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    body()
            g.replay()
        else:
            body()
        torch.cuda.synchronize()
        return [host(t) for t in ys + wins + yv + pools]

    eager, graphed = run(False), run(True)
    for a, b in zip(eager, graphed):
        assert_bits(b, a, "graph vs eager")
    assert sc.get_error() == 0


def test_rollback_layers_equals_per_layer_rollback_and_oracle():
    """One launch for all layers' states gives each layer's rollback."""
    L, N, D, H, K = 3, 21, 5, 256, 3
    s = wl.verify_serving(layers=L, batch=N, D=D, H=H, K=K, n_slots=40, seed=130)
    pools = torch.stack([dev(s.pools[l], "bf16") for l in range(L)])  # [L, n_slots, H, K]
    wins = torch.empty((L, N, D, H, K), dtype=torch.bfloat16, device="cuda")
    slots, acc = dev(s.slot_ids, "i32"), dev(s.accepted, "i32")
    for l in range(L):
        sc.verify(dev(s.bcx[l], "bf16"), dev(s.w[l], "bf16"), slots, pools[l], D, win=wins[l])
    per_layer = pools.clone()
    sc.rollback_layers(wins, acc, slots, pools)
    for l in range(L):
        sc.rollback(wins[l], acc, slots, per_layer[l])
    torch.cuda.synchronize()
    assert_bits(host(pools), host(per_layer), "stacked vs per-layer rollback")
    for l in range(L):
        pool_ref = s.pools[l].copy()
        st, win_ref, _ = oracle.verify("bf16", s.bcx[l], s.w[l], s.slot_ids, pool_ref, D)
        assert st == oracle.OK
        assert oracle.rollback("bf16", win_ref, s.accepted, s.slot_ids, pool_ref) == oracle.OK
        assert_bits(host(pools[l]), pool_ref, f"layer {l} vs oracle")
    assert sc.get_error() == 0


def test_rollback_layers_flags_bad_accepted_once_and_skips_it():
    L, N, D, H, K = 2, 4, 3, 64, 3
    s = wl.verify_serving(layers=L, batch=N, D=D, H=H, K=K, n_slots=8, seed=131)
    pools = torch.stack([dev(s.pools[l], "bf16") for l in range(L)])
    wins = torch.stack([dev(wl.normal(np.random.default_rng(l), (N, D, H, K), 1.0, "bf16"),
                            "bf16") for l in range(L)])
    acc = s.accepted.copy()
    acc[2] = D + 1                                    # out of [0, D]
    before = host(pools)
    sc.rollback_layers(wins, dev(acc, "i32"), dev(s.slot_ids, "i32"), pools)
    assert sc.get_error() == sc.DEV_BAD_ACCEPTED
    after = host(pools)
    bad_slot = s.slot_ids[2]
    assert_bits(after[:, bad_slot], before[:, bad_slot], "skipped sequence's slots")
