"""Bounded waits: a stalled pipeline ends with VS_ERR_TIMEOUT, not a hang.

Every in-kernel wait of the attention kernels gives up after a limit,
records VS_ERR_TIMEOUT in the workspace status block, frees its tensor
memory and returns.  The library's test hook (environment, read by the
launchers) gives the dK / dV kernel's planner, and the producers of a ring
step's query-major kernel, no work: they issue no copy and arrive on no
barrier, so each consumer's first wait runs out after the 2 s limit.  No
copy or MMA is ever in flight when the kernels unwind.  Normal calls
afterwards on the same context must succeed and reproduce the results of
ones made before, bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import f64, inject_index, to_dev

pytestmark = pytest.mark.gpu


def test_stalled_pipeline_times_out_and_context_recovers(monkeypatch):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    w = synth.make_workload(4, L=2048, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.1)
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95)
    ix = inject_index(vs, p, index, dev)
    # a ring of two workers over the striped index (its query-major kernel
    # is the ring-step instance)
    index2, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.1, stripes=2)
    p2 = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95, stripes=2)
    ix2 = inject_index(vs, p2, index2, dev)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    wsf, wsb = vs.workspace(p, vs.VS_OP_FWD, dev), vs.workspace(p, vs.VS_OP_BWD, dev)
    wsr = vs.workspace(p2, vs.VS_OP_RING_FWD, dev)

    def run():
        O = torch.empty_like(Q)
        lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
        vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
        torch.cuda.synchronize()
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
        vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
        O2 = torch.empty_like(Q)
        lse2 = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
        vs.vs_striped_ring_fwd(p2, ix2, Q, K, V, O2, lse2, wsr)
        torch.cuda.synchronize()
        return O, lse, dQ, dK, dV, O2, lse2

    before = run()
    assert all(vs.vs_device_status(ws) == vs.VS_OK for ws in (wsf, wsb, wsr))

    monkeypatch.setenv("VS_TEST_STALL_PRODUCERS", "1")
    run()
    assert vs.vs_device_status(wsb) == vs.VS_ERR_TIMEOUT   # the dK / dV kernels
    assert vs.vs_device_status(wsr) == vs.VS_ERR_TIMEOUT   # the ring steps' forward kernel
    assert vs.vs_device_status(wsf) == vs.VS_OK            # a plain forward carries no hook
    # vs_device_status cleared the status words
    assert vs.vs_device_status(wsb) == vs.VS_OK and vs.vs_device_status(wsr) == vs.VS_OK

    monkeypatch.delenv("VS_TEST_STALL_PRODUCERS")
    after = run()
    assert all(vs.vs_device_status(ws) == vs.VS_OK for ws in (wsf, wsb, wsr))
    for a, b in zip(before, after):
        assert torch.equal(a, b)
