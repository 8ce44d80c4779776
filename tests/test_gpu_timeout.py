"""Bounded waits: a stalled pipeline ends with VS_ERR_TIMEOUT, not a hang.

Every in-kernel wait of the attention kernels gives up after a limit,
records VS_ERR_TIMEOUT in the workspace status block, frees its tensor
memory and returns.  The library's test hook (environment, read by the
launchers and passed to the kernels as a loop bound) gives the producer
warps no work, so they issue no copy and arrive on no barrier, and each
consumer's first wait runs out after the 2 s limit.  No copy or MMA is ever in flight when the kernels unwind.  A normal
call afterwards on the same context must succeed and reproduce the results
of one made before, bit for bit.
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
    w = synth.make_workload(3, L=2048, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.1)
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95)
    ix = inject_index(vs, p, index, dev)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    wsf, wsb = vs.workspace(p, vs.VS_OP_FWD, dev), vs.workspace(p, vs.VS_OP_BWD, dev)

    def run():
        O = torch.empty_like(Q)
        lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
        vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
        vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
        torch.cuda.synchronize()
        return O, lse, dQ, dK, dV

    before = run()
    assert vs.vs_device_status(wsf) == vs.VS_OK and vs.vs_device_status(wsb) == vs.VS_OK

    monkeypatch.setenv("VS_TEST_STALL_PRODUCERS", "1")
    run()
    assert vs.vs_device_status(wsf) == vs.VS_ERR_TIMEOUT
    assert vs.vs_device_status(wsb) == vs.VS_ERR_TIMEOUT
    # vs_device_status cleared the status words
    assert vs.vs_device_status(wsf) == vs.VS_OK and vs.vs_device_status(wsb) == vs.VS_OK

    monkeypatch.delenv("VS_TEST_STALL_PRODUCERS")
    after = run()
    assert vs.vs_device_status(wsf) == vs.VS_OK and vs.vs_device_status(wsb) == vs.VS_OK
    for a, b in zip(before, after):
        assert torch.equal(a, b)
