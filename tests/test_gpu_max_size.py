"""The largest supported sequence, L = 2^20 tokens (GQA 2/1, d = 128).

Index (budget fill to density 0.05): the GPU's masses against the oracle's,
its kept sets exactly equal to the oracle's selection on those masses, and
equal to the oracle's fp64 selection up to ties at the threshold.  Under the
oracle's index: forward on sampled rows against the oracle; backward dQ on
sampled rows and
dK / dV through the identities that hold for any mask (summed over keys, dV
gives the sum of dO over the group's rows and dK gives zero)."""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, budget_sets_agree, f64, gpu_index_lists, inject_index, rel_l2, to_dev

pytestmark = pytest.mark.gpu

L_MAX = 1 << 20


def test_max_length_index_forward_backward():
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    w = synth.make_workload(3, L=L_MAX, Hq=2, Hkv=1, d=128, backward=True)
    density = 0.05
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95, density=density)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    ix = vs.IndexBuffers.allocate(p, dev)
    vs.vs_index_build(p, Q, K, ix, vs.workspace(p, vs.VS_OP_INDEX, dev))
    torch.cuda.synchronize()

    # index: masses, same-precision decisions, and end to end against fp64
    q, k = f64(w.q), f64(w.k)
    v_or, S_or = oracle.index_scores(q, k, 64)
    np.testing.assert_allclose(ix.v_score.double().cpu().numpy(), v_or, rtol=1e-4, atol=1e-12)
    lists = gpu_index_lists(ix, w.Hq)
    act = ix.active_entries.cpu().numpy()
    dens32 = float(np.float32(density))
    index = []
    for h in range(w.Hq):
        v32 = ix.v_score[h].cpu().numpy().astype(np.float64)
        S32 = ix.s_score[h].cpu().numpy().astype(np.float64)
        Vo, So = oracle.select_budget(v32, S32, w.L, 64, dens32)
        np.testing.assert_array_equal(lists[h][0], Vo)
        np.testing.assert_array_equal(lists[h][1], So)
        assert act[h] == oracle.active_entries(w.L, Vo, So, 64)
        kept_or = oracle.select_budget(v_or[h], S_or[h], w.L, 64, dens32)
        ok, bad = budget_sets_agree(v_or[h], S_or[h], kept_or, lists[h])
        assert ok, bad[:5]
        index.append(kept_or)

    # forward then backward (a training step) under the oracle's index
    ix_or = inject_index(vs, p, index, dev)
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    wsf = vs.workspace(p, vs.VS_OP_FWD, dev)
    vs.vs_sparse_attn_fwd(p, ix_or, Q, K, V, O, lse, wsf)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    wsb = vs.workspace(p, vs.VS_OP_BWD, dev)
    vs.vs_sparse_attn_bwd(p, ix_or, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
    torch.cuda.synchronize()
    assert vs.vs_device_status(wsf) == vs.VS_OK and vs.vs_device_status(wsb) == vs.VS_OK

    # forward and dQ on sampled rows (first, middle and last blocks)
    rows = np.concatenate([np.arange(0, 64), np.arange(L_MAX // 2, L_MAX // 2 + 64), np.arange(L_MAX - 64, L_MAX)])
    Or, lser = oracle.attention_forward_rows(q, k, f64(w.v), index, rows)
    sel = torch.from_numpy(rows).to(dev)
    got = f64(bf16_bits_of(O[sel]))
    assert np.abs(got - Or).max() <= 2e-2 and rel_l2(got, Or) <= 1e-2
    assert np.abs(lse.double().cpu().numpy()[:, rows] - lser).max() <= 1e-3
    rQ = oracle.attention_backward_dq_rows(q, k, f64(w.v), f64(w.do), index, rows)
    gq = f64(bf16_bits_of(dQ[sel]))
    assert np.abs(gq - rQ).max() <= 2e-2 * max(1.0, np.abs(rQ).max()) and rel_l2(gq, rQ) <= 1e-2

    # dK / dV identities over all keys
    dVf, dKf = f64(bf16_bits_of(dV)), f64(bf16_bits_of(dK))
    ref = f64(w.do).sum((0, 1))
    got_v = dVf[:, 0].sum(0)
    assert (np.abs(got_v - ref) <= 1e-3 * np.abs(dVf[:, 0]).sum(0) + 1e-2 * np.abs(ref) + 1e-2).all()
    assert (np.abs(dKf[:, 0].sum(0)) <= 1e-3 * np.abs(dKf[:, 0]).sum(0) + 1e-3).all()
