"""Sparse attention backward on the GPU vs the fp64 oracle.

The backward's inputs O and LSE come from the oracle's forward (O rounded
to bf16 as a forward stores it), so that each gradient can be held element
by element to the arithmetic the kernels state: bf16 inputs, fp32
accumulation, P and dS rounded to bf16 where they enter a tensor-core
product, D = rowsum(dO * O) from the bf16 O.  ``grad_close`` checks every
element against that arithmetic (``oracle.attention_backward_bf16_products``)
within 2e-2 + half a bf16 ulp, and against the exact fp64 gradient within the
same plus the arithmetic's own deviation at that element, with relative L2
<= 1e-2.  Both use the same (oracle-built, injected) index.  The chained
forward -> backward of a training step is checked at full size (below and
in test_gpu_max_size.py), where no full oracle backward fits.

Every case runs both ways of forming dQ: from the dS tiles that the dK / dV
pass stores in a workspace with room for them, and by recomputing S and dP
in the minimum workspace; the status word says which one ran.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits_of, f64, grad_close, inject_index, rel_l2, to_dev, ulp_bf16

pytestmark = pytest.mark.gpu


# workspace of the backward: room for every dS block any index can have
# (WS_ALL), room suggested for a budget-fill index of a given density (a
# float), or the minimum (WS_MIN: dS recomputed)
WS_ALL, WS_MIN = "all", None


def _ws_bytes(vs, w, stripes, ws_density):
    """Bytes of a backward workspace (see WS_*).  The dS blocks sit last, so
    room for n blocks per head is the suggested size for density 1 less its
    blocks plus n: nb^2 covers every slash block (nb (nb + 1) / 2) and every
    vertical chunk (at most I per query block I)."""
    mk = lambda dens: vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=stripes,
                                     density=dens)
    if ws_density != WS_ALL:
        return vs.vs_workspace_bytes(mk(ws_density), vs.VS_OP_BWD)
    nb = w.L // 64
    cap1 = int(1.5 * nb * (nb + 1) / 2 + 4 * nb) + 1
    head = vs.vs_workspace_bytes(mk(1.0), vs.VS_OP_BWD) - w.Hq * cap1 * 8192
    return head + w.Hq * nb * nb * 8192


def _fwd_bwd(w, index, stripes=1, density=0.0, O_lse=None, ws_density=WS_ALL, want_path=None, ws_trim=0,
             params_kw=None, want_passes=None):
    """GPU backward; O / LSE from the GPU forward, or injected (O_lse).
    ws_density sizes the backward workspace (see WS_*), less ws_trim bytes
    from its end (the dS blocks sit last); want_path, when given, is the dQ
    path the status word must report (1 stored, 0 recomputed), want_passes
    the number of stored-dS passes; params_kw adds fields of vs_params (e.g.
    rope_mode)."""
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=stripes,
                       density=density, **(params_kw or {}))
    if index is None:
        ix = vs.IndexBuffers.allocate(p, dev)
    else:
        ix = inject_index(vs, p, index, dev)
    Q, K, V, dO = (to_dev(a, dev) for a in (w.q, w.k, w.v, w.do))
    if index is None:
        vs.vs_index_build(p, Q, K, ix, vs.workspace(p, vs.VS_OP_INDEX, dev))
    if O_lse is None:
        O = torch.empty_like(Q)
        lse = torch.empty((w.Hq, w.L), dtype=torch.float32, device=dev)
        wsf = vs.workspace(p, vs.VS_OP_FWD, dev)
        vs.vs_sparse_attn_fwd(p, ix, Q, K, V, O, lse, wsf)
    else:
        O = to_dev(synth.f64_to_bf16_bits(O_lse[0]), dev)
        lse = torch.from_numpy(O_lse[1].astype(np.float32)).to(dev)
        wsf = None
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    if ws_density is WS_MIN:
        wsb = vs.workspace(p, vs.VS_OP_BWD_MIN, dev)
    else:
        wsb = torch.empty(_ws_bytes(vs, w, stripes, ws_density) - ws_trim, dtype=torch.uint8, device=dev)
        assert wsb.numel() > vs.vs_workspace_bytes(p, vs.VS_OP_BWD_MIN)
    vs.vs_sparse_attn_bwd(p, ix, Q, K, V, O, lse, dO, dQ, dK, dV, wsb)
    torch.cuda.synchronize()
    path = int(wsb[8:12].view(torch.int32).item())
    passes = int(wsb[12:16].view(torch.int32).item())
    assert wsf is None or vs.vs_device_status(wsf) == vs.VS_OK
    assert vs.vs_device_status(wsb) == vs.VS_OK
    if want_path is not None:
        assert path == want_path, ("dQ path", path, want_path)
    assert passes == (0 if path == 0 else (want_passes or 1)), ("passes", passes, want_passes)
    return ix, [f64(bf16_bits_of(t)) for t in (dQ, dK, dV)]


def _close(got, ref, name):
    """Chained forward -> backward at full size (sampled rows): max-abs 2e-2
    scaled by the gradient's magnitude and relative L2 1e-2; the forward's
    own bf16 output enters D here, which the injected tests exclude."""
    err = np.abs(got - ref).max()
    rl2 = rel_l2(got, ref)
    bound = 2e-2 * max(1.0, float(np.abs(ref).max()))
    assert err <= bound and rl2 <= 1e-2, (name, err, bound, rl2)


def _check(w, index, stripes=1):
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    O_lse = oracle.attention_forward(q, k, v, index, stripes=stripes)
    ref = oracle.attention_backward(q, k, v, do, index, stripes=stripes)
    emu = oracle.attention_backward_bf16_products(q, k, v, do, index, stripes=stripes)
    for ws_density, path in ((WS_ALL, 1), (WS_MIN, 0)):
        _, got = _fwd_bwd(w, index, stripes, O_lse=O_lse, ws_density=ws_density, want_path=path)
        for name, g, r, e in zip(("dQ", "dK", "dV"), got, ref, emu):
            grad_close(name, g, r, e)


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


def _rope_adjoint(g, kw):
    return oracle.rope(g, kw["rope_theta"], transpose=True, yarn_factor=kw["yarn_factor"],
                       yarn_orig_len=kw["yarn_orig_len"])


def _rope_pair_ulps(src):
    """bf16 ulps of the two channels a rotation mixes into each output
    element: channel i and i + d/2 of the same row."""
    u = ulp_bf16(src)
    h = src.shape[-1] // 2
    both = u[..., :h] + u[..., h:]
    return np.concatenate([both, both], axis=-1)


@pytest.mark.parametrize("yarn", [False, True])
def test_bwd_rope_mode_maps_gradients_back(yarn):
    """rope_mode = 1 returns the gradients of the un-rotated queries and
    keys.  On the stored-dS path the RoPE adjoint of dQ is fused into the dQ
    kernel's epilogue (one rounding); the recomputing path's dQ and every dK
    take the RoPE kernel after the backward.  Each output equals the same
    kernels' rope_mode = 0 gradient rotated back in fp64 (the oracle's RoPE
    adjoint) to the bf16 rounding of the output, plus, for the fused dQ, the
    rotated rounding of its two source channels; dV is unchanged bit for bit;
    relative L2 to the rotated exact gradient <= 1e-2."""
    w = synth.make_workload(3, L=1024, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.1)
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    O_lse = oracle.attention_forward(q, k, v, index)
    ref = oracle.attention_backward(q, k, v, do, index)
    kw = dict(rope_theta=1e4, yarn_factor=4.0 if yarn else 1.0, yarn_orig_len=256 if yarn else 0)
    m = oracle.rope_mscale(kw["yarn_factor"])
    for ws_density, path in ((WS_ALL, 1), (WS_MIN, 0)):
        _, g0 = _fwd_bwd(w, index, O_lse=O_lse, ws_density=ws_density, want_path=path, params_kw=kw)
        _, g1 = _fwd_bwd(w, index, O_lse=O_lse, ws_density=ws_density, want_path=path,
                         params_kw=dict(kw, rope_mode=1))
        for name, a, b, fused in (("dQ", g0[0], g1[0], path == 1), ("dK", g0[1], g1[1], False)):
            want = _rope_adjoint(a, kw)
            bound = 0.5 * ulp_bf16(want) + 2e-6 * m * np.abs(a).max()
            if fused:
                bound = bound + 0.5 * m * _rope_pair_ulps(a)
            err = np.abs(b - want)
            assert (err <= bound).all(), (name, path, float((err - bound).max()))
        np.testing.assert_array_equal(g1[2], g0[2])
        for name, got, r in (("dQ", g1[0], ref[0]), ("dK", g1[1], ref[1])):
            assert rel_l2(got, _rope_adjoint(r, kw)) <= 1e-2, (name, path)


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


def test_bwd_production_shape_element_wise():
    """Element-wise dQ / dK / dV at a production-like shape: GQA 4 / 1,
    L = 16384, budget fill to 5 % density.  The vertical units split their
    rows 32 ways and the slash units add the fp32 partials in their epilogue,
    as at L = 131072."""
    w = synth.make_workload(3, L=16384, Hq=4, Hkv=1, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.05)
    assert max(len(V) for V, _ in index) > 0 and max(len(S) for _, S in index) > 1
    _check(w, index)


def test_bwd_stored_ds_overflow_falls_back():
    """A workspace with room for fewer dS blocks than the index needs: the
    device-side plan finds that a head's blocks do not fit, nothing is
    stored, and dQ is recomputed (status path 0) with the same results."""
    w = synth.make_workload(3, L=2048, Hq=4, Hkv=2, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=0.05)
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    O_lse = oracle.attention_forward(q, k, v, index)
    # room for density 1e-6 is four vertical chunks per query block and one
    # block per head; trimmed to two blocks per head (band 0 alone needs 32)
    nb = w.L // 64
    trim = (4 * nb - 1) * w.Hq * 64 * 64 * 2
    _, got = _fwd_bwd(w, index, O_lse=O_lse, ws_density=1e-6, want_path=0, ws_trim=trim)
    ref = oracle.attention_backward(q, k, v, do, index)
    emu = oracle.attention_backward_bf16_products(q, k, v, do, index)
    for name, g, r, e in zip(("dQ", "dK", "dV"), got, ref, emu):
        grad_close(name, g, r, e)


@pytest.mark.parametrize("Hq,Hkv,hpp,passes", [(8, 4, 2, 4), (6, 3, 4, 2), (3, 3, 1, 3), (16, 2, 8, 2)])
def test_bwd_stored_ds_in_passes(Hq, Hkv, hpp, passes):
    """A workspace whose dS room holds the expected blocks of hpp heads
    only: the backward runs in passes over key/value head groups (4, 2 with
    an uneven last pass, 3 with unpaired heads, 2), every pass on the stored
    path; gradients against the oracle, and the same bits as one pass with
    room for every head."""
    dens = 0.3
    w = synth.make_workload(3, L=2048, Hq=Hq, Hkv=Hkv, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=dens)
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    O_lse = oracle.attention_forward(q, k, v, index)
    # the suggested room gives every head cap blocks; keep hpp heads' worth
    nb = w.L // 64
    cap = int(1.5 * dens * nb * (nb + 1) / 2 + 4 * nb) + 1
    trim = (w.Hq - hpp) * cap * 64 * 64 * 2
    _, got = _fwd_bwd(w, index, density=dens, O_lse=O_lse, ws_density=dens, want_path=1, ws_trim=trim,
                      want_passes=passes)
    _, one = _fwd_bwd(w, index, density=dens, O_lse=O_lse, ws_density=dens, want_path=1)
    ref = oracle.attention_backward(q, k, v, do, index)
    emu = oracle.attention_backward_bf16_products(q, k, v, do, index)
    for name, g, o, r, e in zip(("dQ", "dK", "dV"), got, one, ref, emu):
        grad_close(name, g, r, e)
        np.testing.assert_array_equal(g, o, err_msg=name)


def test_bwd_stored_ds_passes_rope_mode_striped():
    """Four stored-dS passes with rope_mode = 1 (the RoPE adjoint of dQ in
    the epilogue of every pass's dQ kernel, dK's after the last pass) on
    striped tiles (W = 2): the same bits as one pass."""
    dens = 0.3
    w = synth.make_workload(4, L=2048, Hq=8, Hkv=4, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, stripes=2, density=dens)
    q, k, v = f64(w.q), f64(w.k), f64(w.v)
    O_lse = oracle.attention_forward(q, k, v, index, stripes=2)
    nb = w.L // 64
    cap = int(1.5 * dens * nb * (nb + 1) / 2 + 4 * nb) + 1
    kw = dict(rope_mode=1, rope_theta=1e4)
    _, got = _fwd_bwd(w, index, stripes=2, density=dens, O_lse=O_lse, ws_density=dens, want_path=1,
                      ws_trim=(w.Hq - 2) * cap * 64 * 64 * 2, params_kw=kw, want_passes=4)
    _, one = _fwd_bwd(w, index, stripes=2, density=dens, O_lse=O_lse, ws_density=dens, want_path=1, params_kw=kw)
    for name, g, o in zip(("dQ", "dK", "dV"), got, one):
        np.testing.assert_array_equal(g, o, err_msg=name)


def test_bwd_striped_32_shards():
    w = synth.make_workload(4, L=4096, Hq=2, Hkv=1, d=128, backward=True)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.9, stripes=32)
    _check(w, index, stripes=32)


def test_bwd_full_size_gqa_128k():
    """The 128K GQA training workload at full size under the oracle's
    budget-fill index (forward then backward on the GPU, as in a training
    step): dQ on sampled rows and dK / dV of the keys of two blocks near the
    end against the oracle, all keys' dK / dV through identities that hold
    for any mask (keys summed: dV -> sum of dO over the group's rows,
    dK -> 0)."""
    w = synth.make_workload(3)
    index, _, _ = oracle.build_index(f64(w.q), f64(w.k), 64, 0.95, density=float(np.float32(0.05)))
    rows = np.concatenate([np.arange(0, 64), np.arange(65536, 65536 + 64), np.arange(w.L - 64, w.L)])
    q, k, v, do = f64(w.q), f64(w.k), f64(w.v), f64(w.do)
    rQ = oracle.attention_backward_dq_rows(q, k, v, do, index, rows)
    # dK / dV of the keys of two blocks near the end (few rows reach them)
    nb = w.L // 64
    keys = np.concatenate([np.arange((nb - 8) * 64, (nb - 7) * 64), np.arange((nb - 1) * 64, nb * 64)])
    rK, rV = oracle.attention_backward_dkdv_keys(q, k, v, do, index, keys)
    # the bench's workspace (room for the dS tiles of density 0.05), then the minimum
    for ws_density, path in ((0.05, 1), (WS_MIN, 0)):
        ix, (dQ, dK, dV) = _fwd_bwd(w, index, ws_density=ws_density, want_path=path)
        _check_full(w, dQ, dK, dV, rows, rQ)
        _close(dK[keys], rK, "dK keys")
        _close(dV[keys], rV, "dV keys")


def _check_full(w, dQ, dK, dV, rows, rQ):
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
