"""Sparse attention backward on the GPU vs the fp64 oracle.

The GPU forward supplies O and LSE (as a training step would); the oracle
differentiates its own exact fp64 masked attention.  Both use the same
(oracle-built, injected) index.

Tolerance (bf16 in, fp32 accumulation): relative L2 <= 1e-2, and max-abs
<= 2e-2 scaled by max(1, max |ref|).  The scale factor is needed because the
gradients are not unit-scale: dQ reaches ~17 and dV ~30 on these inputs (6x
norm outlier keys that take almost all of a row's softmax mass), and a bf16
value near 16 has a rounding step of 1/16 by storage alone.  The arithmetic
is FlashAttention's: D = rowsum(dO * O) from the bf16 O, and P / dS rounded to
bf16 for the tensor-core products; an fp64 emulation of exactly that
arithmetic gives the same errors as the GPU to two digits.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, f64, inject_index, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _fwd_bwd(w, index, stripes=1, density=0.0):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=stripes,
                       density=density)
    if index is None:
        ix = vs.IndexBuffers.allocate(p, dev)
    else:
        ix = inject_index(vs, p, index, dev)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    if index is None:
        vs.vs_index_build(p, Q, K, ix, vs.workspace(p, vs.VS_OP_INDEX, dev))
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    wsf = vs.workspace(p, vs.VS_OP_FWD, dev)
    vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    wsb = vs.workspace(p, vs.VS_OP_BWD, dev)
    vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
    torch.cuda.synchronize()
    assert vs.vs_device_status(wsf) == vs.VS_OK
    assert vs.vs_device_status(wsb) == vs.VS_OK
    return ix, [f64(bf16_bits_of(t)) for t in (dQ, dK, dV)]


def _close(got, ref, name):
    err = np.abs(got - ref).max()
    rl2 = rel_l2(got, ref)
    bound = 2e-2 * max(1.0, float(np.abs(ref).max()))
    assert err <= bound and rl2 <= 1e-2, (name, err, bound, rl2)


def _check(w, index, stripes=1):
    _, (dQ, dK, dV) = _fwd_bwd(w, index, stripes)
    rQ, rK, rV = oracle.attention_backward(f64(w.q), f64(w.k), f64(w.v), f64(w.do), index, stripes=stripes)
    _close(dQ, rQ, "dQ")
    _close(dK, rK, "dK")
    _close(dV, rV, "dV")


CASES = [
    # wid, L, Hq, Hkv, top_p   (d = 128)
    (3, 256, 2, 1, 0.9),
    (3, 1024, 4, 2, 0.5),
    (3, 1024, 4, 2, 0.95),
    (3, 2048, 16, 2, 0.9),
    (3, 512, 1, 1, 0.9),      # same-head tiles
    (3, 320, 3, 1, 0.7),      # odd group size, odd block count
    (2, 1024, 4, 4, 0.9),
]


@pytest.mark.parametrize("wid,L,Hq,Hkv,p_", CASES)
def test_bwd_topp_index(wid, L, Hq, Hkv, p_):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=128, top_p=p_, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), w.last_q, p_)
    _check(w, index)


def test_bwd_budget_fill_index():
    w = synth.make_workload(3, L=2048, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.05)
    _check(w, index)


@pytest.mark.parametrize("name", ["only_diag", "all_bands", "all_verts", "last_vert", "mixed"])
@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (1, 1)])
def test_bwd_edge_masks(name, Hq, Hkv):
    L = 512
    nb = L // 64
    rng = np.random.default_rng(3)
    idx = dict(
        only_diag=[(np.array([], np.int64), np.array([0]))] * Hq,
        all_bands=[(np.array([], np.int64), np.arange(nb))] * Hq,
        all_verts=[(np.arange(L), np.array([0]))] * Hq,
        last_vert=[(np.array([L - 1, 5]), np.array([0, 2]))] * Hq,
        mixed=[(np.sort(rng.choice(L, 40, replace=False)), np.union1d(rng.choice(nb, 3, replace=False), [0]))
               for _ in range(Hq)],
    )[name]
    w = synth.make_workload(3, L=L, Hq=Hq, Hkv=Hkv, d=128, backward=True)
    _check(w, idx)


def test_bwd_striped_bands():
    w = synth.make_workload(4, L=2048, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.9, stripes=4)
    _check(w, index, stripes=4)


def test_bwd_striped_32_shards():
    w = synth.make_workload(4, L=4096, Hq=2, Hkv=1, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.9, stripes=32)
    _check(w, index, stripes=32)


def test_bwd_full_size_gqa_128k():
    """The 128K GQA training workload at full size with the GPU budget-fill
    index: dQ on sampled rows against the oracle, dK / dV through identities
    that hold for any mask (keys summed: dV -> sum of dO over the group's
    rows, dK -> 0)."""
    from _util import gpu_index_lists
    w = synth.make_workload(3)
    ix, (dQ, dK, dV) = _fwd_bwd(w, None, density=0.05)
    index = gpu_index_lists(ix, w.Hq)
    rows = np.concatenate([np.arange(0, 64), np.arange(65536, 65536 + 64), np.arange(w.L - 64, w.L)])
    rQ = oracle.attention_backward_dq_rows(f64(w.q), f64(w.k), f64(w.v), f64(w.do), index, rows)
    _close(dQ[rows], rQ, "dQ rows")
    G = w.Hq // w.Hkv
    dOf = f64(w.do)
    for g in range(w.Hkv):
        ref = dOf[:, g * G:(g + 1) * G].sum((0, 1))
        got = dV[:, g].sum(0)
        # bf16 rounding of each row adds a random-walk error ~ eps * sqrt(L)
        # of the rows' magnitude; a real error scales with the L1 mass
        l1v = np.abs(dV[:, g]).sum(0)
        assert (np.abs(got - ref) <= 1e-3 * l1v + 1e-2 * np.abs(ref) + 1e-2).all()
        l1k = np.abs(dK[:, g]).sum(0)
        assert (np.abs(dK[:, g].sum(0)) <= 1e-3 * l1k + 1e-3).all()
