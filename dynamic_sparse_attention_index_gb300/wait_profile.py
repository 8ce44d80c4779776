"""Pipeline-balance timers of the attention kernels (diagnostic).

The attention kernels can be built with in-kernel cycle counters
(``VS_WAIT_PROFILE=<mode>`` in the environment of the build): the counts land
in the ``wait_cycles`` array of the device status block at the head of the
call's workspace.  This module runs one forward and one backward call on the
GQA 16/2, d = 128 synthetic workload and prints the counters per tile.

Light modes (per-thread register accumulation, little perturbation):
  4  dK/dV kernel: MMA-thread issue time of S/dP and of dV/dK
  6  query-major kernel (forward, dQ): MMA issue time of S, dP and the
     accumulate, the role warps' waits, and each softmax warp's wait / work
     split

Usage (from the repository root, on a GPU):

    VS_WAIT_PROFILE=6 python -m dynamic_sparse_attention_index_gb300.wait_profile --L 131072
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

SLOTS = {
    "4": {24: "MMA issue S / dP", 25: "MMA issue dV / dK"},
    "6": {0: "MMA issue S", 9: "MMA issue dP", 19: "MMA issue accumulate (P V or dS K)",
          1: "K producer waits q_empty", 2: "K producer waits k_empty", 3: "K producer waits meta_free",
          4: "V producer waits v_empty", 7: "K producer total", 8: "V producer total",
          10: "MMA waits p_ready", 11: "MMA waits o_free", 12: "MMA waits k_full", 13: "MMA waits q_full",
          14: "MMA waits dp_free", 15: "MMA waits v_full", 5: "MMA metadata copy (+ q_full)",
          6: "MMA K release commit",
          21: "softmax warp: waits for metadata and S", 27: "softmax warp: S -> P / dS written",
          30: "softmax warp: epilogue"},
}
PER_WARP = {21, 27, 30}   # summed over the 8 softmax warps of a CTA


def main() -> None:
    mode = os.environ.get("VS_WAIT_PROFILE", "")
    if mode not in SLOTS:
        sys.exit("build and run with VS_WAIT_PROFILE=4 or 6")
    ap = argparse.ArgumentParser()
    ap.add_argument("--L", type=int, default=32768)
    args = ap.parse_args()
    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import synth
    import dynamic_sparse_attention_index_gb300 as vs
    from dynamic_sparse_attention_index_gb300 import build

    build.build()
    dev = torch.device("cuda:0")
    w = synth.make_workload(3, L=args.L)
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95, density=0.05)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V, dO = (bf(a) for a in (w.q, w.k, w.v, w.do))
    ix = vs.IndexBuffers.allocate(p, dev)
    vs.vs_index_build(p, Q, K, ix, vs.workspace(p, vs.VS_OP_INDEX, dev))
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    wsf, wsb = vs.workspace(p, vs.VS_OP_FWD, dev), vs.workspace(p, vs.VS_OP_BWD, dev)
    for _ in range(2):
        vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
        vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
    torch.cuda.synchronize()
    calls = [("backward (dK/dV kernel)", wsb)] if mode == "4" else [("forward", wsf), ("backward (dQ kernel)", wsb)]
    for tag, ws in calls:
        ws[:16 + 32 * 8].zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if ws is wsf:
            vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
        else:
            vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
        e1.record()
        torch.cuda.synchronize()
        c = ws[16:16 + 32 * 8].cpu().numpy().view(np.uint64).astype(np.float64)
        tiles = c[16]
        print(f"== {tag}: {e0.elapsed_time(e1):.3f} ms, {tiles:.0f} tiles, "
              f"{c[31] / tiles:.0f} SM cycles per tile" if tiles else f"== {tag}: no tiles counted")
        for k, name in SLOTS[mode].items():
            if c[k] and tiles:
                per = c[k] / tiles / (8 if k in PER_WARP else 1)
                print(f"   {name:44s} {per:8.0f} cycles per tile{' (per warp)' if k in PER_WARP else ''}")


if __name__ == "__main__":
    main()
