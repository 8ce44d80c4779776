"""Index build on the GPU vs the oracle.

Three levels:
  * scores: the vertical / slash masses match the fp64 oracle's to fp32
    accuracy;
  * decisions: the oracle's selection run on the GPU's own fp32 masses gives
    exactly the GPU's kept sets (both decide in the same precision), and the
    exact active-entry count matches;
  * end to end: the GPU's sets equal the oracle's fp64 sets except for
    elements at the top-p threshold (within 1e-6 normalised mass).
"""
import numpy as np
import pytest

import oracle
import synth
from _util import budget_sets_agree, f64, gpu_index_lists, to_dev, topp_sets_agree

pytestmark = pytest.mark.gpu


def _run(w, density=0.0, stripes=1):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=stripes,
                       density=density)
    Q, K = to_dev(w.q, dev), to_dev(w.k, dev)
    ix = vs.IndexBuffers.allocate(p, dev)
    ws = vs.workspace(p, vs.VS_OP_INDEX, dev)
    vs.vs_index_build(p, Q, K, ix, ws)
    torch.cuda.synchronize()
    return p, ix


CASES = [
    # (workload recipe, L, Hq, Hkv, d, last_q, top_p, stripes)
    (1, 4096, 1, 1, 64, 64, 0.9, 1),
    (1, 256, 1, 1, 64, 64, 0.9, 1),
    (3, 1024, 4, 2, 128, 64, 0.95, 1),
    (3, 2048, 16, 2, 128, 64, 0.5, 1),
    (3, 1024, 4, 1, 64, 16, 0.9, 1),
    (3, 1024, 2, 2, 128, 100, 0.9, 1),
    (3, 4096, 4, 2, 128, 64, 0.95, 4),
    (2, 2048, 8, 8, 128, 64, 1.0, 1),
    (3, 512, 2, 1, 64, 1, 0.9, 1),
    (3, 768, 8, 1, 128, 200, 0.9, 2),
    (4, 4096, 2, 1, 128, 64, 0.9, 32),   # the striped workload's 32 shards
    (3, 2048, 6, 2, 128, 64, 0.9, 1),    # tensor-core scoring, a group of three: one pair holds one head
]


@pytest.mark.parametrize("wid,L,Hq,Hkv,d,lq,p_,W", CASES)
def test_index_topp(wid, L, Hq, Hkv, d, lq, p_, W):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d, last_q=lq, top_p=p_)
    p, ix = _run(w, stripes=W)
    v_or, S_or = oracle.index_scores(f64(w.q), f64(w.k), lq, stripes=W)
    v_gpu = ix.v_score.double().cpu().numpy()
    S_gpu = ix.s_score.double().cpu().numpy()
    np.testing.assert_allclose(v_gpu, v_or, rtol=5e-5, atol=1e-7 * lq / L)
    np.testing.assert_allclose(S_gpu, S_or, rtol=5e-5, atol=1e-7 * lq)
    lists = gpu_index_lists(ix, Hq)
    act = ix.active_entries.cpu().numpy()
    bs = 64 * W
    for h in range(Hq):
        Vg, Sg = lists[h]
        # same-precision decisions: oracle selection on the GPU's fp32 masses
        v32 = ix.v_score[h].cpu().numpy().astype(np.float64)
        S32 = ix.s_score[h].cpu().numpy().astype(np.float64)
        Vo = oracle.select_top_p(v32, np.float32(p_))
        So = np.union1d(oracle.select_top_p(S32, np.float32(p_)), [0])
        np.testing.assert_array_equal(Vg, Vo)
        np.testing.assert_array_equal(Sg, So)
        assert act[h] == oracle.active_entries(L, Vo, So, bs)
        # end to end against the fp64 oracle, ties at the threshold excepted
        ok, bad = topp_sets_agree(v_or[h], oracle.select_top_p(v_or[h], p_), Vg, p_)
        assert ok, bad[:5]
        ok, bad = topp_sets_agree(S_or[h], oracle.select_top_p(S_or[h], p_), Sg, p_, forced=(0,))
        assert ok, bad[:5]


@pytest.mark.parametrize("density", [0.05, 0.2, 0.6])
@pytest.mark.parametrize("wid,L,Hq,Hkv,d,W", [(3, 2048, 4, 2, 128, 1), (1, 4096, 1, 1, 64, 1),
                                              (3, 4096, 2, 1, 128, 2)])
def test_index_budget_fill(wid, L, Hq, Hkv, d, W, density):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d)
    p, ix = _run(w, density=density, stripes=W)
    lists = gpu_index_lists(ix, Hq)
    act = ix.active_entries.cpu().numpy()
    dens32 = float(np.float32(density))
    bs = 64 * W
    for h in range(Hq):
        v32 = ix.v_score[h].cpu().numpy().astype(np.float64)
        S32 = ix.s_score[h].cpu().numpy().astype(np.float64)
        Vo, So = oracle.select_budget(v32, S32, L, bs, dens32)
        np.testing.assert_array_equal(lists[h][0], Vo)
        np.testing.assert_array_equal(lists[h][1], So)
        assert act[h] == oracle.active_entries(L, Vo, So, bs)
        assert act[h] >= dens32 * oracle.total_causal_entries(L)
    # end to end against the fp64 oracle (fp64 masses), ties at the threshold excepted
    v_or, S_or = oracle.index_scores(f64(w.q), f64(w.k), w.last_q, stripes=W)
    for h in range(Hq):
        kept_or = oracle.select_budget(v_or[h], S_or[h], L, bs, dens32)  # the density the call passed
        ok, bad = budget_sets_agree(v_or[h], S_or[h], kept_or, lists[h])
        assert ok, bad[:5]


# The selection kernel's budget fill first gathers the verticals above a
# histogram cut (bins of the fp32 bit pattern >> 20, at most 1024 verticals
# above the cut) and the bands above it (at most 6144); when the set at that
# cut reaches the target it finishes on those lists, otherwise it searches
# bit by bit over the full list.  _select_path repeats that decision on the
# host from the kernel's own masses so a test can show which branch ran.
_FAST_CAP, _BAND_CAP = 1024, 6144


def _select_path(v32, S32, L, bs, density):
    kv = np.asarray(v32, np.float32).view(np.uint32).astype(np.int64)
    ks = np.asarray(S32, np.float32).view(np.uint32).astype(np.int64)
    hist = np.bincount(np.minimum(kv >> 20, 2047), minlength=2048)
    suf = np.append(np.cumsum(hist[::-1])[::-1], 0)
    t_low = int(np.flatnonzero(suf <= _FAST_CAP)[0]) << 20
    Vs = np.flatnonzero(kv >= t_low)
    Ss = np.concatenate([[0], 1 + np.flatnonzero(ks[1:] >= t_low)])
    if len(Ss) - 1 > _BAND_CAP:
        return "bitwise"
    reach = oracle.active_entries(L, Vs, Ss, bs) >= density * oracle.total_causal_entries(L)
    return "fast" if reach else "bitwise"


def _concentrated_workload(L, Hq, Hkv, d, n_heavy, gain):
    """The last queries attend to the first n_heavy keys: a shared direction
    of norm ``gain`` is added to those keys and to the last 64 queries.  The
    slash bands that meet only the other keys then carry almost no mass."""
    w = synth.make_workload(1, L=L, Hq=Hq, Hkv=Hkv, d=d)
    q, k = synth.bf16_bits_to_f64(w.q), synth.bf16_bits_to_f64(w.k)
    u = np.full(d, gain / np.sqrt(d))
    k[:n_heavy] += u
    q[-64:] += u
    w.q, w.k = synth.f64_to_bf16_bits(q), synth.f64_to_bf16_bits(k)
    return w


@pytest.mark.parametrize("density,path", [(0.01, "fast"), (0.2, "fast"), (0.6, "bitwise"),
                                          (0.9, "bitwise")])
def test_index_budget_fill_paths(density, path):
    """Both branches of the budget fill, on an input whose far bands are
    nearly empty: the kept sets equal the oracle's selection on the kernel's
    fp32 masses and the active counts are exact."""
    w = _concentrated_workload(4096, 2, 1, 64, 1200, 10.0)
    p, ix = _run(w, density=density)
    lists = gpu_index_lists(ix, w.Hq)
    act = ix.active_entries.cpu().numpy()
    dens32 = float(np.float32(density))
    for h in range(w.Hq):
        v32 = ix.v_score[h].cpu().numpy().astype(np.float64)
        S32 = ix.s_score[h].cpu().numpy().astype(np.float64)
        assert _select_path(v32, S32, w.L, 64, dens32) == path
        Vo, So = oracle.select_budget(v32, S32, w.L, 64, dens32)
        np.testing.assert_array_equal(lists[h][0], Vo)
        np.testing.assert_array_equal(lists[h][1], So)
        assert act[h] == oracle.active_entries(w.L, Vo, So, 64)
        if density == 0.01:
            assert len(Vo) == 0 and So.tolist() == [0]  # band 0 alone reaches 1 %


def test_index_full_size_gqa_128k():
    """The 128K GQA workload (16 query heads, 2 KV heads, d=128) at full size."""
    w = synth.make_workload(3, backward=False)
    p, ix = _run(w)
    v_or, S_or = oracle.index_scores(f64(w.q), f64(w.k), w.last_q)
    np.testing.assert_allclose(ix.v_score.double().cpu().numpy(), v_or, rtol=1e-4, atol=1e-10)
    np.testing.assert_allclose(ix.s_score.double().cpu().numpy(), S_or, rtol=1e-4, atol=1e-10)
    lists = gpu_index_lists(ix, w.Hq)
    for h in range(w.Hq):
        ok, bad = topp_sets_agree(v_or[h], oracle.select_top_p(v_or[h], w.top_p), lists[h][0], w.top_p)
        assert ok, bad[:5]
        ok, bad = topp_sets_agree(S_or[h], oracle.select_top_p(S_or[h], w.top_p), lists[h][1], w.top_p,
                                  forced=(0,))
        assert ok, bad[:5]
        assert 0 in lists[h][1].tolist()
        # planted outliers carry most of the mass: all of them are verticals
        assert set(w.outliers.tolist()) <= set(lists[h][0].tolist())
    # the measured operating point: budget fill to 5 % density, end to end
    # against the oracle's fp64 selection, and the exact active counts
    _, ixb = _run(w, density=0.05)
    listsb = gpu_index_lists(ixb, w.Hq)
    act = ixb.active_entries.cpu().numpy()
    for h in range(w.Hq):
        kept_or = oracle.select_budget(v_or[h], S_or[h], w.L, 64, float(np.float32(0.05)))
        ok, bad = budget_sets_agree(v_or[h], S_or[h], kept_or, listsb[h])
        assert ok, bad[:5]
        if all(np.array_equal(a, b) for a, b in zip(kept_or, listsb[h])):
            assert act[h] == oracle.active_entries(w.L, kept_or[0], kept_or[1], 64)


@pytest.mark.parametrize("wid,L,Hq,Hkv,d,W,dens", [(3, 2048, 8, 2, 128, 1, 0.0), (3, 4096, 16, 2, 128, 1, 0.05),
                                                  (1, 4096, 1, 1, 64, 1, 0.0), (4, 4096, 4, 1, 128, 4, 0.0),
                                                  (3, 2048, 6, 2, 64, 1, 0.2)])
def test_index_group_shared(wid, L, Hq, Hkv, d, W, dens):
    """index_mode = 1: each head's lists are exactly the union of its group's
    per-head lists of the same call in per-head mode (same masses, same
    decisions), the active counts are the union's, and the union equals the
    oracle's fp64 group union except for per-head threshold ties."""
    import dynamic_sparse_attention_index_gb300 as vs
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d)
    G = Hq // Hkv
    p0, ix0 = _run(w, density=dens, stripes=W)
    import torch
    dev = torch.device("cuda:0")
    p1 = vs.make_params(w.L, w.Hq, w.Hkv, w.d, last_q=w.last_q, top_p=w.top_p, stripes=W, density=dens,
                        index_mode=vs.VS_INDEX_GROUP_SHARED)
    Q, K = to_dev(w.q, dev), to_dev(w.k, dev)
    ix1 = vs.IndexBuffers.allocate(p1, dev)
    vs.vs_index_build(p1, Q, K, ix1, vs.workspace(p1, vs.VS_OP_INDEX, dev))
    torch.cuda.synchronize()
    per, grp = gpu_index_lists(ix0, Hq), gpu_index_lists(ix1, Hq)
    assert torch.equal(ix0.v_score, ix1.v_score) and torch.equal(ix0.s_score, ix1.s_score)
    union = oracle.group_shared_index(per, G)
    act = ix1.active_entries.cpu().numpy()
    bs = 64 * W
    for h in range(Hq):
        np.testing.assert_array_equal(grp[h][0], union[h][0])
        np.testing.assert_array_equal(grp[h][1], union[h][1])
        assert act[h] == oracle.active_entries(L, union[h][0], union[h][1], bs)
    # end to end: the fp64 oracle's union, differences only at per-head ties
    v_or, S_or = oracle.index_scores(f64(w.q), f64(w.k), w.last_q, stripes=W)
    idx_or, _, _ = oracle.build_index(f64(w.q), f64(w.k), w.last_q, w.top_p, stripes=W,
                                      density=float(np.float32(dens)) if dens else 0.0)
    shared_or = oracle.group_shared_index(idx_or, G)
    for g in range(Hkv):
        dv = set(shared_or[g * G][0].tolist()) ^ set(grp[g * G][0].tolist())
        ds = set(shared_or[g * G][1].tolist()) ^ set(grp[g * G][1].tolist())
        for h in range(g * G, (g + 1) * G):
            if dens:
                ok, bad = budget_sets_agree(v_or[h], S_or[h], idx_or[h], per[h])
            else:
                ok = topp_sets_agree(v_or[h], idx_or[h][0], per[h][0], w.top_p)[0] and \
                     topp_sets_agree(S_or[h], idx_or[h][1], per[h][1], w.top_p, forced=(0,))[0]
            assert ok
        tie_v = set().union(*[set(idx_or[h][0].tolist()) ^ set(per[h][0].tolist()) for h in range(g * G, (g + 1) * G)])
        tie_s = set().union(*[set(idx_or[h][1].tolist()) ^ set(per[h][1].tolist()) for h in range(g * G, (g + 1) * G)])
        assert dv <= tie_v and ds <= tie_s
