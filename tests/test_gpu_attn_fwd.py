"""Sparse attention forward on the GPU vs the fp64 oracle.

Both sides use the same index (the oracle's, injected into the device
buffers) so that top-p ties cannot leak into the output comparison.
Tolerance (bf16 inputs, fp32 accumulation, P rounded to bf16 for P V):
max-abs <= 2e-2 and relative L2 <= 1e-2 on O; LSE within 1e-3 absolute.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, f64, inject_index, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _fwd(w, index, stripes=1):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=stripes)
    ix = inject_index(vs, p, index, dev)
    Q, K, V = to_dev(w.q, dev), to_dev(w.k, dev), to_dev(w.v, dev)
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    ws = vs.workspace(p, vs.VS_OP_FWD, dev)
    vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, ws)
    torch.cuda.synchronize()
    assert vs.vs_device_status(ws) == vs.VS_OK
    return f64(bf16_bits_of(O)), lse.double().cpu().numpy()


def _check(w, index, stripes=1, rows=None):
    O, lse = _fwd(w, index, stripes)
    if rows is None:
        Or, lser = oracle.attention_forward(f64(w.q), f64(w.k), f64(w.v), index, stripes=stripes)
        got, glse = O, lse
    else:
        Or, lser = oracle.attention_forward_rows(f64(w.q), f64(w.k), f64(w.v), index, rows, stripes=stripes)
        got, glse = O[rows], lse[:, rows]
    assert np.abs(got - Or).max() <= 2e-2
    assert rel_l2(got, Or) <= 1e-2
    assert np.abs(glse - lser).max() <= 1e-3


CASES = [
    # wid, L, Hq, Hkv, d, top_p
    (1, 256, 1, 1, 64, 0.9),
    (1, 4096, 1, 1, 64, 0.9),
    (3, 512, 2, 1, 128, 0.9),
    (3, 1024, 4, 2, 128, 0.5),
    (3, 1024, 4, 2, 64, 0.95),
    (3, 2048, 16, 2, 128, 0.9),
    (2, 1024, 4, 4, 128, 0.9),
    (3, 192, 1, 1, 128, 0.9),     # odd block count, same-head tiles
    (3, 320, 3, 1, 64, 0.7),      # odd group size
]


@pytest.mark.parametrize("wid,L,Hq,Hkv,d,p_", CASES)
def test_fwd_topp_index(wid, L, Hq, Hkv, d, p_):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d, top_p=p_)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), w.last_q, p_)
    _check(w, index)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_budget_fill_index(d):
    w = synth.make_workload(3, L=2048, Hq=4, Hkv=2, d=d)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.05)
    _check(w, index)


def _edge_indices(L, Hq):
    nb = L // 64
    rng = np.random.default_rng(3)
    only_diag = [(np.array([], np.int64), np.array([0]))] * Hq
    all_bands = [(np.array([], np.int64), np.arange(nb))] * Hq
    all_verts = [(np.arange(L), np.array([0]))] * Hq
    last_vert = [(np.array([L - 1, 5]), np.array([0, 2]))] * Hq
    mixed = []
    for h in range(Hq):
        S = np.union1d(rng.choice(nb, 3, replace=False), [0])
        V = np.sort(rng.choice(L, 40, replace=False))      # many fall inside kept bands
        mixed.append((V, S))
    return dict(only_diag=only_diag, all_bands=all_bands, all_verts=all_verts, last_vert=last_vert,
                mixed=mixed)


@pytest.mark.parametrize("name", ["only_diag", "all_bands", "all_verts", "last_vert", "mixed"])
@pytest.mark.parametrize("Hq,Hkv,d", [(2, 1, 128), (1, 1, 64)])
def test_fwd_edge_masks(name, Hq, Hkv, d):
    w = synth.make_workload(3, L=512, Hq=Hq, Hkv=Hkv, d=d)
    _check(w, _edge_indices(512, Hq)[name])


def test_fwd_striped_bands():
    w = synth.make_workload(4, L=2048, Hq=4, Hkv=2, d=128)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.9, stripes=4)
    _check(w, index, stripes=4)


def test_fwd_striped_32_shards():
    """The striped-layout workload's 32 round-robin shards: slash tiles of
    64 x 32 tokens (two bands at L = 4096)."""
    w = synth.make_workload(4, L=4096, Hq=2, Hkv=1, d=128)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.9, stripes=32)
    _check(w, index, stripes=32)


def test_fwd_full_size_gqa_128k_sampled():
    """The 128K GQA workload at full size under the oracle's budget-fill
    index, checked on sampled rows (first, middle, last blocks; every head)."""
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    w = synth.make_workload(3, backward=False)
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95, density=0.05)
    Q, K, V = to_dev(w.q, dev), to_dev(w.k, dev), to_dev(w.v, dev)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=float(np.float32(0.05)))
    ix = inject_index(vs, p, index, dev)
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    ws = vs.workspace(p, vs.VS_OP_FWD, dev)
    vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, ws)
    torch.cuda.synchronize()
    assert vs.vs_device_status(ws) == vs.VS_OK
    rows = np.concatenate([np.arange(0, 70), np.arange(65536 - 3, 65536 + 67), np.arange(w.L - 70, w.L)])
    Or, lser = oracle.attention_forward_rows(f64(w.q), f64(w.k), f64(w.v), index, rows)
    got = f64(bf16_bits_of(O[torch.from_numpy(rows).to(dev)]))
    assert np.abs(got - Or).max() <= 2e-2
    assert rel_l2(got, Or) <= 1e-2
    assert np.abs(lse.double().cpu().numpy()[:, rows] - lser).max() <= 1e-3


@pytest.mark.parametrize("Hq,Hkv,lo,hi", [(4, 2, 512, 1536), (3, 1, 256, 768), (2, 1, 0, 2048)])
def test_fwd_row_range(Hq, Hkv, lo, hi):
    """vs_sparse_attn_fwd_rows: the rows of a context-parallel worker.  Its
    rows are bit-identical to the full call's (each row tile is computed the
    same way whichever others run) and the other rows stay untouched."""
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    w = synth.make_workload(3, L=2048, Hq=Hq, Hkv=Hkv, d=128)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.1)
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95)
    ix = inject_index(vs, p, index, dev)
    Q, K, V = to_dev(w.q, dev), to_dev(w.k, dev), to_dev(w.v, dev)
    ws = vs.workspace(p, vs.VS_OP_FWD, dev)
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, ws)
    O2 = torch.full_like(Q, 7.0)
    lse2 = torch.full((w.Hq, w.L), 7.0, dtype=torch.float32, device=dev)
    vs.vs_sparse_attn_fwd_rows(p, ix, Q, K, V, O2, lse2, ws, lo, hi)
    torch.cuda.synchronize()
    # odd group sizes work on pairs of 64-row blocks: widen to whole pairs
    if (Hq // Hkv) % 2:
        lo, hi = lo // 128 * 128, (hi + 127) // 128 * 128
    assert torch.equal(O2[lo:hi], O[lo:hi]) and torch.equal(lse2[:, lo:hi], lse[:, lo:hi])
    assert (O2[:lo] == 7.0).all() and (O2[hi:] == 7.0).all()
    assert (lse2[:, :lo] == 7.0).all() and (lse2[:, hi:] == 7.0).all()
