"""The largest supported sequence, L = 2^20 tokens (GQA 2/1, d = 128), and
the 512K GQA shape whose stored dS tiles take several passes.

Index (budget fill to density 0.05): the GPU's masses against the oracle's,
its kept sets exactly equal to the oracle's selection on those masses, and
equal to the oracle's fp64 selection up to ties at the threshold.  Under the
oracle's index: forward on sampled rows against the oracle; backward dQ on
sampled rows and dK / dV of the keys of two blocks near the end against the
oracle, and all keys' dK / dV through the identities that hold for any mask
(summed over keys, dV gives the sum of dO over the group's rows and dK gives
zero)."""
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

    # dK / dV of the keys of two blocks near the end against the oracle
    nb = L_MAX // 64
    keys = np.concatenate([np.arange((nb - 8) * 64, (nb - 7) * 64), np.arange((nb - 1) * 64, nb * 64)])
    rK, rV = oracle.attention_backward_dkdv_keys(q, k, f64(w.v), f64(w.do), index, keys)
    sk = torch.from_numpy(keys).to(dev)
    for name, got, ref in (("dK", f64(bf16_bits_of(dK[sk])), rK), ("dV", f64(bf16_bits_of(dV[sk])), rV)):
        assert np.abs(got - ref).max() <= 2e-2 * max(1.0, np.abs(ref).max()) and rel_l2(got, ref) <= 1e-2, name

    # dK / dV identities over all keys
    dVf, dKf = f64(bf16_bits_of(dV)), f64(bf16_bits_of(dK))
    ref = f64(w.do).sum((0, 1))
    got_v = dVf[:, 0].sum(0)
    assert (np.abs(got_v - ref) <= 1e-3 * np.abs(dVf[:, 0]).sum(0) + 1e-2 * np.abs(ref) + 1e-2).all()
    assert (np.abs(dKf[:, 0].sum(0)) <= 1e-3 * np.abs(dKf[:, 0]).sum(0) + 1e-3).all()


def test_512k_stored_ds_in_passes():
    """L = 524288 with GQA 8 / 2 (four query heads per key/value head, as
    the 512K 32 / 8 workload), budget fill to density 0.05: 20.9 GB of dS
    blocks per head, so the suggested workspace (78 GiB) holds one group at
    a time and the backward stores the tiles in two passes.  dK and dV are
    the same bits as with dQ recomputed (the same dK / dV kernels ran); dQ
    of both paths on sampled rows, and dK / dV of the keys of two blocks near
    the end, against the oracle (under the GPU's own index); dV summed over
    all keys against the identity that holds for any mask.  (The matching
    identity for dK, a zero sum, is not checked here: D is formed from the
    forward's bf16 output, whose products took P in bf16, and where outlier
    keys at 8x put most of a row's softmax on one key that makes D differ
    from the P . dP of the backward by ~1e-2, so such a row's dS sums to
    that instead of zero; 2M rows add it up beyond any slack that would
    still catch an error.)"""
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    w = synth.make_workload(5, Hq=8, Hkv=2, backward=True)
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=64, top_p=0.95, density=0.05)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    ix = vs.IndexBuffers.allocate(p, dev)
    vs.vs_index_build(p, Q, K, ix, vs.workspace(p, vs.VS_OP_INDEX, dev))
    O = torch.empty_like(Q)
    lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
    wsf = vs.workspace(p, vs.VS_OP_FWD, dev)
    vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
    grads = {}
    for op, path, passes in ((vs.VS_OP_BWD, 1, 2), (vs.VS_OP_BWD_MIN, 0, 0)):
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
        wsb = vs.workspace(p, op, dev)
        vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
        torch.cuda.synchronize()
        assert vs.vs_device_status(wsf) == vs.VS_OK and vs.vs_device_status(wsb) == vs.VS_OK
        st = wsb[:16].view(torch.int32).cpu().numpy()
        assert (int(st[2]), int(st[3])) == (path, passes), st
        grads[path] = (dQ, bf16_bits_of(dK), bf16_bits_of(dV))
        del wsb
        torch.cuda.empty_cache()
    np.testing.assert_array_equal(grads[1][1], grads[0][1])
    np.testing.assert_array_equal(grads[1][2], grads[0][2])

    # dQ on sampled rows; only those rows of Q and dO are converted (the
    # rest of the fp64 arrays stay untouched zero pages)
    index = gpu_index_lists(ix, w.Hq)
    rows = np.concatenate([np.arange(0, 64), np.arange(w.L // 2, w.L // 2 + 64), np.arange(w.L - 64, w.L)])
    q = np.zeros((w.L, w.Hq, w.d))
    do = np.zeros((w.L, w.Hq, w.d))
    q[rows], do[rows] = f64(w.q[rows]), f64(w.do[rows])
    k64, v64 = f64(w.k), f64(w.v)
    rQ = oracle.attention_backward_dq_rows(q, k64, v64, do, index, rows)
    sel = torch.from_numpy(rows).to(dev)
    for path in (1, 0):
        gq = f64(bf16_bits_of(grads[path][0][sel]))
        err = np.abs(gq - rQ)
        print(f"\n512K dQ path {path}: max |err| {err.max():.3g} (max |dQ| {np.abs(rQ).max():.3g}),"
              f" relative L2 {rel_l2(gq, rQ):.3g}")
        # chained forward -> backward (as the other full-size checks): the
        # bound scales with the gradient's magnitude (here up to ~40, where
        # the bf16 P and dS of the products alone move an element by ~2^-9
        # of it besides its own half-ulp rounding); the element-wise tests
        # hold the tight bound against the bf16-products oracle
        assert err.max() <= 2e-2 * max(1.0, np.abs(rQ).max()) and rel_l2(gq, rQ) <= 1e-2, path

    # dK / dV of two key blocks near the end (the rows reaching them are the
    # last 512 and, for a vertical among them, the rows after it)
    nb = w.L // 64
    keys = np.concatenate([np.arange((nb - 8) * 64, (nb - 7) * 64), np.arange((nb - 1) * 64, nb * 64)])
    tail = np.arange(w.L - 512, w.L)
    q[tail], do[tail] = f64(w.q[tail]), f64(w.do[tail])
    rK, rV = oracle.attention_backward_dkdv_keys(q, k64, v64, do, index, keys)
    for name, got, ref in (("dK", f64(grads[1][1][keys]), rK), ("dV", f64(grads[1][2][keys]), rV)):
        err = np.abs(got - ref)
        print(f"512K {name} keys: max |err| {err.max():.3g} (max |{name}| {np.abs(ref).max():.3g}),"
              f" relative L2 {rel_l2(got, ref):.3g}")
        assert err.max() <= 2e-2 * max(1.0, np.abs(ref).max()) and rel_l2(got, ref) <= 1e-2, name

    # dV summed over all keys equals dO summed over the group's rows (softmax
    # rows sum to one), per key/value head
    G = w.Hq // w.Hkv
    dVf = f64(grads[1][2])
    for g in range(w.Hkv):
        ref = np.zeros(w.d)
        for r0 in range(0, w.L, 1 << 16):
            ref += f64(w.do[r0:r0 + (1 << 16), g * G:(g + 1) * G]).sum((0, 1))
        got_v = dVf[:, g].sum(0)
        assert (np.abs(got_v - ref) <= 1e-3 * np.abs(dVf[:, g]).sum(0) + 1e-2 * np.abs(ref) + 1e-2).all()
