"""Striped sparse ring attention on the GPU (W workers, W steps each, run
one after another with a carried softmax state) against the oracle.

The oracle's ring (``oracle.striped_ring_forward``) is pinned equal to the
single-pass masked attention under the striped index, so the GPU ring is
compared with the single-pass oracle functions, element by element, with the
tolerances of the single-launch tests: forward max-abs 2e-2, relative L2
1e-2, LSE 1e-3; backward (from the oracle's O and LSE) every element within
2e-2 + half a bf16 ulp of the bf16-products oracle and relative L2 1e-2 of
the exact one.  Per-step CUDA events are recorded and must all complete.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, f64, grad_close, inject_index, rel_l2, to_dev, ulp_bf16

pytestmark = pytest.mark.gpu


def _ring(w, W, index, O_lse=None, events=False, params_kw=None):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=w.top_p, stripes=W, **(params_kw or {}))
    ix = inject_index(vs, p, index, dev)
    Q, K, V = to_dev(w.q, dev), to_dev(w.k, dev), to_dev(w.v, dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(W * W + 1)] if events else None
    out = {}
    if O_lse is None:
        O = torch.empty_like(Q)
        lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
        ws = vs.workspace(p, vs.VS_OP_RING_FWD, dev)
        vs.vs_striped_ring_fwd(p, ix, Q, K, V, O, lse, ws, events=ev)
        torch.cuda.synchronize()
        assert vs.vs_device_status(ws) == vs.VS_OK
        out["O"], out["lse"] = f64(bf16_bits_of(O)), lse.double().cpu().numpy()
    else:
        dO = to_dev(w.do, dev)
        O = to_dev(synth.f64_to_bf16_bits(O_lse[0]), dev)
        lse = torch.from_numpy(O_lse[1].astype(np.float32)).to(dev)
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
        ws = vs.workspace(p, vs.VS_OP_RING_BWD, dev)
        vs.vs_striped_ring_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, ws, events=ev)
        torch.cuda.synchronize()
        assert vs.vs_device_status(ws) == vs.VS_OK
        out["grads"] = [f64(bf16_bits_of(t)) for t in (dQ, dK, dV)]
    if events:
        t = [ev[k].elapsed_time(ev[k + 1]) for k in range(W * W)]
        assert all(x >= 0 for x in t)
        out["steps_ms"] = np.array(t).reshape(W, W)
    return out


CASES = [
    # wid, L, Hq, Hkv, d, W, top_p, density
    (4, 2048, 4, 2, 128, 4, 0.9, 0.0),
    (4, 4096, 2, 1, 128, 32, 0.9, 0.0),     # the striped workload's 32 shards (128 local rows each)
    (4, 8192, 4, 2, 128, 4, 0.95, 0.05),    # budget fill
    (4, 2048, 3, 1, 128, 2, 0.7, 0.0),      # odd group size: same-head tiles
    (3, 1024, 2, 1, 128, 1, 0.9, 0.0),      # one worker: the plain call
]


@pytest.mark.parametrize("wid,L,Hq,Hkv,d,W,p_,dens", CASES)
def test_ring_forward_backward(wid, L, Hq, Hkv, d, W, p_, dens):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d, top_p=p_, backward=True)
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    index, _, _ = oracle.build_index(q, k, 64, p_, stripes=W, density=dens)
    Or, lser = oracle.attention_forward(q, k, v, index, stripes=W)
    got = _ring(w, W, index, events=True)
    assert np.abs(got["O"] - Or).max() <= 2e-2
    assert rel_l2(got["O"], Or) <= 1e-2
    assert np.abs(got["lse"] - lser).max() <= 1e-3
    assert got["steps_ms"].shape == (W, W)
    g = _ring(w, W, index, O_lse=(Or, lser))["grads"]
    ref = oracle.attention_backward(q, k, v, do, index, stripes=W)
    emu = oracle.attention_backward_bf16_products(q, k, v, do, index, stripes=W)
    for name, a, r, e in zip(("dQ", "dK", "dV"), g, ref, emu):
        grad_close(name, a, r, e)


def test_ring_backward_rope_mode():
    """rope_mode = 1 on the ring: dQ and dK come back through the RoPE
    adjoint (the RoPE kernel after the ring), equal to the rope_mode = 0
    gradients rotated back in fp64 to the bf16 rounding of the output; dV
    unchanged bit for bit."""
    w = synth.make_workload(4, L=2048, Hq=4, Hkv=2, d=128, top_p=0.9, backward=True)
    q, k, v = f64(w.q), f64(w.k), f64(w.v)
    index, _, _ = oracle.build_index(q, k, 64, 0.9, stripes=4)
    O_lse = oracle.attention_forward(q, k, v, index, stripes=4)
    kw = dict(rope_theta=1e4, yarn_factor=1.0, yarn_orig_len=0)
    g0 = _ring(w, 4, index, O_lse=O_lse, params_kw=kw)["grads"]
    g1 = _ring(w, 4, index, O_lse=O_lse, params_kw=dict(kw, rope_mode=1))["grads"]
    for name, a, b in (("dQ", g0[0], g1[0]), ("dK", g0[1], g1[1])):
        want = oracle.rope(a, 1e4, transpose=True)
        err = np.abs(b - want)
        bound = 0.5 * ulp_bf16(want) + 2e-6 * np.abs(a).max()
        assert (err <= bound).all(), (name, float((err - bound).max()))
    np.testing.assert_array_equal(g1[2], g0[2])


def test_ring_forward_d64():
    w = synth.make_workload(4, L=2048, Hq=2, Hkv=1, d=64)
    q, k, v = f64(w.q), f64(w.k), f64(w.v)
    index, _, _ = oracle.build_index(q, k, 64, 0.9, stripes=4)
    Or, lser = oracle.attention_forward(q, k, v, index, stripes=4)
    got = _ring(w, 4, index)
    assert np.abs(got["O"] - Or).max() <= 2e-2 and rel_l2(got["O"], Or) <= 1e-2
    assert np.abs(got["lse"] - lser).max() <= 1e-3


def test_ring_edge_masks():
    """Only the diagonal band (the first local row of every tile sees no key
    in the steps whose shard comes after the worker's), and every band."""
    L, W = 2048, 4
    nb = L // (64 * W)
    w = synth.make_workload(4, L=L, Hq=2, Hkv=1, d=128, backward=True)
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    for index in ([(np.array([], np.int64), np.array([0]))] * 2,
                  [(np.array([3, 700, 1500]), np.arange(nb))] * 2):
        Or, lser = oracle.attention_forward(q, k, v, index, stripes=W)
        got = _ring(w, W, index)
        assert np.abs(got["O"] - Or).max() <= 2e-2 and np.abs(got["lse"] - lser).max() <= 1e-3
        g = _ring(w, W, index, O_lse=(Or, lser))["grads"]
        ref = oracle.attention_backward(q, k, v, do, index, stripes=W)
        emu = oracle.attention_backward_bf16_products(q, k, v, do, index, stripes=W)
        for name, a, r, e in zip(("dQ", "dK", "dV"), g, ref, emu):
            grad_close(name, a, r, e)
