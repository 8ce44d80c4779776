"""Anti-diagonal block scorer on the GPU vs the oracle.

  * scores: the GPU's block scores match the fp64 oracle's to fp32 accuracy;
  * decisions: the oracle's selection run on the GPU's own fp32 scores gives
    exactly the GPU's kept blocks (both decide in the same precision), and
    the kept-block counts and active entries are exact;
  * at the 128K GQA shape: sampled block rows of the oracle, the same two
    checks on them;
  * recall and sparsity against the vertical-slash index on the same input
    (contiguous and striped tiles), measured with the oracle's exact
    attention mass on sampled rows.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle.vs_oracle import _row_mask
from _util import f64, to_dev

pytestmark = pytest.mark.gpu


def _run(w, stride, thr, stripes=1):
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    dev = torch.device("cuda:0")
    p = vs.make_params(w.L, w.Hq, w.Hkv, w.d, stripes=stripes)
    Q, K = to_dev(w.q, dev), to_dev(w.k, dev)
    ix = vs.XattnBuffers.allocate(p, dev)
    ws = vs.workspace(p, vs.VS_OP_XATTN, dev)
    vs.vs_xattn_index_build(p, stride, thr, Q, K, ix, ws)
    torch.cuda.synchronize()
    assert vs.vs_device_status(ws) == vs.VS_OK
    return p, ix


def _check_decisions(ix, X32, thr, bs, rows=None):
    """The oracle's selection on the GPU's fp32 scores equals the GPU's."""
    kept = ix.kept_blocks()
    cnt = ix.block_cnt.cpu().numpy()
    Hq, nb = cnt.shape
    rows = list(range(nb)) if rows is None else list(rows)
    want = oracle.xattn_select(X32, thr, block_rows=rows)
    for h in range(Hq):
        for n, I in enumerate(rows):
            np.testing.assert_array_equal(kept[h][I], want[h][n], err_msg=f"head {h} block row {I}")
            assert cnt[h, I] == len(want[h][n])
    return kept


CASES = [
    # (workload recipe, L, Hq, Hkv, d, stride, stripes, threshold)
    (3, 1024, 2, 1, 128, 8, 1, 0.9),
    (3, 1600, 2, 2, 64, 8, 1, 0.9),     # 200 strided rows: a ragged last row tile
    (3, 2048, 4, 2, 128, 4, 1, 0.8),    # 16 strided rows per block
    (1, 2048, 3, 1, 64, 16, 1, 0.95),   # 4 per block, odd group
    (3, 1024, 2, 1, 128, 1, 1, 0.9),    # stride 1: exact block masses, 64-row blocks
    (3, 2048, 1, 1, 128, 1, 2, 0.9),    # 128-row blocks
    (3, 1024, 2, 2, 64, 1, 1, 0.9),     # d = 64 with 64-row blocks
    (4, 4096, 2, 1, 128, 8, 4, 0.9),    # striped tiles, bs = 256
    (3, 4096, 2, 1, 128, 8, 1, 1.0),    # threshold 1: every block of positive score
    (4, 8192, 2, 1, 128, 16, 32, 0.9),  # the 32-stripe tile, bs = 2048: 128 strided rows per block
    (4, 8192, 2, 1, 64, 32, 32, 0.9),   # 64 per block
]


@pytest.mark.parametrize("wid,L,Hq,Hkv,d,S,W,thr", CASES)
def test_xattn_scores_and_selection(wid, L, Hq, Hkv, d, S, W, thr):
    w = synth.make_workload(wid, L=L, Hq=Hq, Hkv=Hkv, d=d, stripes=W)
    p, ix = _run(w, S, thr, stripes=W)
    bs = 64 * W
    X_or = oracle.xattn_block_scores(f64(w.q), f64(w.k), S, bs)
    X_gpu = ix.block_score.double().cpu().numpy()
    np.testing.assert_allclose(X_gpu, X_or, rtol=1e-4, atol=1e-7)
    # every block row sums to one, nothing above the diagonal
    np.testing.assert_allclose(X_gpu.sum(axis=2), 1.0, rtol=1e-4)
    nb = L // bs
    iu = np.triu_indices(nb, 1)
    assert np.all(X_gpu[:, iu[0], iu[1]] == 0)
    X32 = ix.block_score.cpu().numpy().astype(np.float64)
    kept = _check_decisions(ix, X32, np.float32(thr), bs)
    act = ix.active_entries.cpu().numpy()
    for h in range(Hq):
        assert act[h] == oracle.xattn_active_entries(kept[h], bs)
    if thr >= 1.0:
        for h in range(Hq):
            for I in range(nb):
                np.testing.assert_array_equal(kept[h][I], np.flatnonzero(X32[h, I, :I + 1] > 0))


def test_xattn_full_size_gqa_128k_sampled_rows():
    """The 128K GQA workload (16 query heads, 2 key/value heads, d = 128),
    stride 8: sampled block rows (first, last, and between) of two heads of
    different groups against the oracle."""
    w = synth.make_workload(3, backward=False)
    p, ix = _run(w, 8, 0.9)
    rows = [0, 1, 37, 1024, 1500, 2047]
    heads = [0, 9]
    Xs = ix.block_score[heads][:, rows, :].double().cpu().numpy()
    # heads 0 and 9 use key/value heads 0 and 1: with the two query heads
    # alone, the oracle pairs query head i with key/value head i
    X_or = oracle.xattn_block_scores(f64(w.q[:, heads, :]), f64(w.k), 8, 64, block_rows=rows)
    np.testing.assert_allclose(Xs, X_or, rtol=1e-4, atol=1e-8)
    kept = ix.kept_blocks()
    want = oracle.xattn_select(Xs.astype(np.float32).astype(np.float64), np.float32(0.9), block_rows=rows)
    for n, h in enumerate(heads):
        for m, I in enumerate(rows):
            np.testing.assert_array_equal(kept[h][I], want[n][m])
    act = ix.active_entries.cpu().numpy()
    cnt = ix.block_cnt.cpu().numpy()
    for h in range(w.Hq):
        assert act[h] == int(((cnt[h] - 1) * 64 * 64).sum()) + (w.L // 64) * (64 * 65 // 2)
        assert (cnt[h] >= 1).all() and (cnt[h] <= np.arange(1, w.L // 64 + 1)).all()


@pytest.mark.parametrize("W", [1, 4])
def test_xattn_recall_and_sparsity_vs_vertical_slash(W, capsys):
    """Recall (exact attention mass on the kept entries, sampled rows) and
    sparsity of the anti-diagonal block index at thresholds 0.1, 0.5 and 0.9,
    each against the vertical-slash index filled to the same density, on the
    128K workload's distributions at L = 8192 (16 / 2 heads shrunk to 4 / 1)."""
    import torch
    import dynamic_sparse_attention_index_gb300 as vs
    from _util import gpu_index_lists
    L, bs = 8192, 64 * W
    w = synth.make_workload(3, L=L, Hq=4, Hkv=1, d=128, stripes=W, backward=False)
    dev = torch.device("cuda:0")
    Q, K = to_dev(w.q, dev), to_dev(w.k, dev)
    q, k = f64(w.q), f64(w.k)
    rows = np.arange(37, L, 97)
    total = oracle.total_causal_entries(L) * w.Hq
    lines = []
    for thr in (0.1, 0.5, 0.9):
        p, ix = _run(w, 8, thr, stripes=W)
        act_x = int(ix.active_entries.sum())
        pv = vs.make_params(L, w.Hq, w.Hkv, w.d, stripes=W, density=float(act_x / total))
        vix = vs.IndexBuffers.allocate(pv, dev)
        vs.vs_index_build(pv, Q, K, vix, vs.workspace(pv, vs.VS_OP_INDEX, dev))
        torch.cuda.synchronize()
        lists = gpu_index_lists(vix, w.Hq)
        act_v = int(vix.active_entries.sum())
        kept = ix.kept_blocks()
        rec_x = oracle.attention_recall(q, k, lambda h, r: oracle.xattn_row_mask(r, L, kept[h], bs), rows)
        rec_v = oracle.attention_recall(q, k, lambda h, r: _row_mask(r, L, lists[h][0], lists[h][1], bs), rows)
        lines.append(f"W={W} threshold {thr}: anti-diagonal recall {rec_x:.4f} at sparsity {1 - act_x / total:.4f};"
                     f" vertical-slash recall {rec_v:.4f} at sparsity {1 - act_v / total:.4f}")
        # budget fill reaches the requested density per head (rounded to fp32)
        assert act_v >= act_x * (1 - 1e-6)
        assert 0.0 < rec_x <= 1.0 + 1e-9 and 0.0 < rec_v <= 1.0 + 1e-9
    with capsys.disabled():
        print("\n" + "\n".join(lines))
