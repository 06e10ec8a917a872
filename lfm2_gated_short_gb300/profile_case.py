"""Run a few launches of one ShortConv call on a seeded case, for profilers.

    python -m lfm2_gated_short_gb300.profile_case prefill  --T 4096 --launches 6
    python -m lfm2_gated_short_gb300.profile_case decode   --N 256  --launches 6
    python -m lfm2_gated_short_gb300.profile_case verify   --N 64 --D 8 --launches 6
    python -m lfm2_gated_short_gb300.profile_case rollback --N 64 --D 8 --layers 10 --launches 3
    python -m lfm2_gated_short_gb300.profile_case backward --T 65536 --launches 3
    python -m lfm2_gated_short_gb300.profile_case backward_varlen --T 65536 --seqs 57 --launches 3
    python -m lfm2_gated_short_gb300.profile_case in_proj  --T 4096 --seqs 16 --launches 3
    python -m lfm2_gated_short_gb300.profile_case out_proj --T 4096 --launches 3
    python -m lfm2_gated_short_gb300.profile_case in_proj_decode --N 256 --launches 6

Inputs are drawn on the device with a seeded generator (bf16, N(0,1) data,
N(0,1/3) weights, N(0,1) pools). Consecutive launches rotate over three input
sets so that a launch does not find the previous one's data in L2 for the
full-size cases. Exits non-zero if the library reports a device error.
"""
from __future__ import annotations

import argparse

import torch

import lfm2_gated_short_gb300 as sc


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["prefill", "prefill_tiled", "decode", "verify", "rollback",
                                   "backward", "backward_varlen", "in_proj", "out_proj",
                                   "in_proj_decode"])
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--H", type=int, default=2048)
    ap.add_argument("--K", type=int, default=3)
    ap.add_argument("--N", type=int, default=256)
    ap.add_argument("--D", type=int, default=8)
    ap.add_argument("--slots", type=int, default=1024)
    ap.add_argument("--tile", type=int, default=8)
    ap.add_argument("--seqs", type=int, default=None,
                    help="packed sequences: backward_varlen (default 16), in_proj (default 1)")
    ap.add_argument("--layers", type=int, default=10, help="stacked layers (rollback)")
    ap.add_argument("--launches", type=int, default=6)
    a = ap.parse_args()
    if a.seqs is None:
        a.seqs = 16 if a.op == "backward_varlen" else 1
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(7)

    def rnd(*shape, std=1.0):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    H, K = a.H, a.K
    w = rnd(H, K, std=(1 / 3) ** 0.5)
    Dm = H  # model width of the projections (LFM2-1.2B: D = H)
    w_in = rnd(3 * H, Dm, std=Dm ** -0.5) if a.op in ("in_proj", "in_proj_decode") else None
    w_out = rnd(Dm, H, std=H ** -0.5) if a.op == "out_proj" else None
    sets = []
    for _ in range(3):
        if a.op in ("prefill", "prefill_tiled"):
            sets.append(dict(bcx=rnd(a.T, 3 * H), y=torch.empty(a.T, H, dtype=torch.bfloat16,
                                                                 device=dev),
                             pool=torch.zeros(1, H, K, dtype=torch.bfloat16, device=dev)))
        elif a.op == "decode":
            sets.append(dict(bcx=rnd(a.N, 3 * H), pool=rnd(a.slots, H, K)))
        elif a.op == "verify":
            sets.append(dict(bcx=rnd(a.N * a.D, 3 * H), pool=rnd(a.slots, H, K)))
        elif a.op == "rollback":  # every layer's verify tape, then one stacked rollback
            sets.append(dict(win=rnd(a.layers, a.N, a.D, H, K),
                             pools=rnd(a.layers, a.slots, H, K)))
        elif a.op == "in_proj":
            sets.append(dict(hidden=rnd(a.T, Dm), y=torch.empty(a.T, H, dtype=torch.bfloat16,
                                                                 device=dev),
                             pool=rnd(a.slots, H, K)))
        elif a.op == "out_proj":
            sets.append(dict(y=rnd(a.T, H)))
        elif a.op == "in_proj_decode":  # one token for each of N sequences
            sets.append(dict(hidden=rnd(a.N, Dm), pool=rnd(a.slots, H, K)))
        else:
            sets.append(dict(bcx=rnd(a.T, 3 * H), dy=rnd(a.T, H)))
    cu = torch.tensor([0, a.T], dtype=torch.int32, device=dev)
    if a.op in ("backward_varlen", "in_proj"):  # seeded cut points: a.seqs packed sequences
        cuts = torch.randperm(a.T - 1, generator=torch.Generator().manual_seed(7))[:a.seqs - 1] + 1
        cu = torch.cat([torch.tensor([0]), cuts.sort().values, torch.tensor([a.T])]).to(
            torch.int32).to(dev)
        init = rnd(a.seqs, H, K)
    slot0 = torch.zeros(1, dtype=torch.int32, device=dev)
    seq_slots = torch.randperm(a.slots, generator=torch.Generator().manual_seed(8))[:a.seqs].to(
        torch.int32).to(dev)
    slots = torch.randperm(a.slots, generator=torch.Generator().manual_seed(7))[:a.N].to(
        torch.int32).to(dev)
    accepted = torch.randint(0, a.D + 1, (a.N,), generator=torch.Generator().manual_seed(7),
                             dtype=torch.int32).to(dev)
    for i in range(a.launches):
        s = sets[i % 3]
        if a.op == "prefill":
            sc.prefill(s["bcx"], w, cu, slot0, s["pool"], y=s["y"])
        elif a.op == "prefill_tiled":
            sc.prefill(s["bcx"], w, cu, slot0, s["pool"], y=s["y"], rows_per_thread=a.tile)
        elif a.op == "decode":
            sc.decode(s["bcx"], w, slots, s["pool"])
        elif a.op == "verify":
            sc.verify(s["bcx"], w, slots, s["pool"], a.D)
        elif a.op == "rollback":
            sc.rollback_layers(s["win"], accepted, slots, s["pools"])
        elif a.op == "in_proj":
            sc.in_proj_prefill(s["hidden"], w_in, w, cu, seq_slots, s["pool"], y=s["y"])
        elif a.op == "out_proj":
            sc.out_proj(s["y"], w_out)
        elif a.op == "in_proj_decode":
            sc.in_proj_decode(s["hidden"], w_in, w, slots, s["pool"])
        elif a.op == "backward_varlen":
            sc.backward_varlen(s["bcx"], w, cu, s["dy"], init_states=init)
        else:
            sc.backward(s["bcx"], w, s["dy"])
    torch.cuda.synchronize()
    code = sc.get_error()
    if code:
        raise SystemExit(f"device error word {code:#x}")
    print(f"{a.op}: {a.launches} launches ok")


if __name__ == "__main__":
    main()
