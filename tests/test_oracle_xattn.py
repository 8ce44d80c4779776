"""Pins of the anti-diagonal block scorer's oracle against things other than
itself: brute force over the anti-diagonal entries on tiny inputs, the
stride-1 case against a library softmax of the full causal logits, the
row-sum and triangle invariants, a closed form for constant keys, the
selection's recall and minimality, and the active-entry count of an
explicit mask."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _rand(L, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d))


def _brute(Q, K, S, bs):
    """Every cell from the full logit matrix: the entries (i, j) of the S x S
    sub-block with (i - rS) + (j - cS) = S - 1, averaged; softmax and block
    sums by explicit loops."""
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    R, nb = L // S, L // bs
    X = np.zeros((Hq, nb, nb))
    for h in range(Hq):
        lg = (Q[:, h, :] @ K[:, h // G, :].T) / math.sqrt(d)
        for r in range(R):
            z = []
            for c in range(r + 1):
                vals = [lg[i, j] for i in range(r * S, r * S + S) for j in range(c * S, c * S + S)
                        if (i - r * S) + (j - c * S) == S - 1]
                assert len(vals) == S
                z.append(sum(vals) / S)
            mx = max(z)
            e = [math.exp(t - mx) for t in z]
            tot = sum(e)
            for c in range(r + 1):
                X[h, (r * S) // bs, (c * S) // bs] += e[c] / tot
        X[h] *= S / bs
    return X


@pytest.mark.parametrize("L,S,bs,Hq,Hkv,d", [(32, 4, 8, 2, 1, 4), (48, 2, 8, 1, 1, 6), (64, 8, 16, 3, 3, 5),
                                           (32, 1, 8, 2, 2, 3)])
def test_brute_force_anti_diagonals(L, S, bs, Hq, Hkv, d):
    Q, K = _rand(L, Hq, Hkv, d, 7 + L + S)
    np.testing.assert_allclose(oracle.xattn_block_scores(Q, K, S, bs), _brute(Q, K, S, bs), rtol=1e-12, atol=1e-14)


def test_stride_one_is_the_true_block_mass():
    """S = 1: each cell is one entry, so X[I, J] is the causal softmax mass of
    block (I, J) averaged over the block's rows."""
    L, bs, d = 128, 16, 8
    Q, K = _rand(L, 2, 1, d, 3)
    X = oracle.xattn_block_scores(Q, K, 1, bs)
    nb = L // bs
    for h in range(2):
        lg = (Q[:, h, :] @ K[:, 0, :].T) / math.sqrt(d)
        lg[np.triu_indices(L, 1)] = -np.inf
        P = softmax(lg, axis=1)
        ref = P.reshape(nb, bs, nb, bs).sum(axis=(1, 3)) / bs
        np.testing.assert_allclose(X[h], ref, rtol=1e-12, atol=1e-15)


def test_invariants():
    L, S, bs = 512, 8, 64
    Q, K = _rand(L, 2, 1, 16, 11)
    X = oracle.xattn_block_scores(Q, K, S, bs)
    np.testing.assert_allclose(X.sum(axis=2), 1.0, rtol=1e-12)
    assert (X >= 0).all()
    nb = L // bs
    assert np.all(X[:, np.triu_indices(nb, 1)[0], np.triu_indices(nb, 1)[1]] == 0)
    # a subset of block rows gives the same rows
    Xs = oracle.xattn_block_scores(Q, K, S, bs, block_rows=[0, 5, 7])
    np.testing.assert_array_equal(Xs, X[:, [0, 5, 7], :])


def test_constant_keys_closed_form():
    """Equal keys: every kept cell of strided row r has the same score, so
    P[r, c] = 1 / (r + 1) and, with H the harmonic numbers,
    X[I, J] = H((I+1) b) - H(I b) for J < I (b = bs / S strided rows per
    block) and X[I, I] = (1/b) sum_{r in I} (r - I b + 1) / (r + 1)."""
    L, S, bs, d = 256, 4, 32, 8
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((L, 1, d))
    K = np.tile(rng.standard_normal((1, 1, d)), (L, 1, 1))
    X = oracle.xattn_block_scores(Q, K, S, bs)[0]
    b, nb = bs // S, L // bs
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, L // S + 1))])
    for I in range(nb):
        for J in range(I):
            assert X[I, J] == pytest.approx(H[(I + 1) * b] - H[I * b], rel=1e-12)
        diag = sum((r - I * b + 1) / (r + 1) for r in range(I * b, (I + 1) * b)) / b
        assert X[I, I] == pytest.approx(diag, rel=1e-12)


@pytest.mark.parametrize("p", [0.3, 0.7, 0.9, 0.999])
def test_selection_recall_and_minimality(p):
    """Each row's kept blocks reach p of its mass with the diagonal forced;
    dropping the smallest kept block other than the diagonal falls below p
    (unless the diagonal alone reaches it); ties never split a kept value."""
    L, S, bs = 1024, 8, 64
    Q, K = _rand(L, 2, 1, 32, 21)
    X = oracle.xattn_block_scores(Q, K, S, bs)
    kept = oracle.xattn_select(X, p)
    for h in range(2):
        for I, J in enumerate(kept[h]):
            row = X[h, I, :I + 1]
            assert I in J.tolist() and np.all(np.diff(J) > 0) and J.max() <= I
            free = [j for j in J.tolist() if j != I]
            # the top-p part alone (without the forced diagonal) reaches p
            sel = oracle.select_top_p(row, p)
            assert row[sel].sum() >= p * row.sum() * (1 - 1e-12)
            assert set(free) <= set(sel.tolist())
            if len(sel) > 1:
                smallest = sel[np.argmin(row[sel])]
                assert row[sel].sum() - row[smallest] < p * row.sum()
            # no unselected block beats a selected one
            if len(sel) < I + 1:
                rest = np.setdiff1d(np.arange(I + 1), sel)
                assert row[rest].max() <= row[sel].min()


def test_threshold_one_keeps_every_positive_block():
    L, S, bs = 256, 4, 32
    Q, K = _rand(L, 1, 1, 8, 2)
    X = oracle.xattn_block_scores(Q, K, S, bs)
    kept = oracle.xattn_select(X, 1.0)
    for I, J in enumerate(kept[0]):
        np.testing.assert_array_equal(J, np.arange(I + 1))


def test_active_entries_and_row_mask_against_explicit_count():
    L, bs = 256, 32
    nb = L // bs
    rng = np.random.default_rng(9)
    kept = [np.union1d(rng.choice(I + 1, size=rng.integers(0, I + 1), replace=False), [I]) for I in range(nb)]
    dense = np.zeros((L, L), bool)
    for n in range(L):
        for m in range(n + 1):
            dense[n, m] = (m // bs) in set(kept[n // bs].tolist())
    assert oracle.xattn_active_entries(kept, bs) == int(dense.sum())
    np.testing.assert_array_equal(oracle.xattn_row_mask(np.arange(L), L, kept, bs), dense)


def test_recall_of_full_mask_is_one_and_block_mass_matches():
    L, bs, d = 256, 32, 8
    Q, K = _rand(L, 2, 1, d, 4)
    rows = np.arange(0, L, 7)
    full = lambda h, r: np.ones((r.size, L), bool)
    assert oracle.attention_recall(Q, K, full, rows) == pytest.approx(1.0, rel=1e-12)
    # recall of a block index = the stride-1 block scores of its kept blocks
    # (stride 1 scores are exact block masses averaged over a block's rows)
    X = oracle.xattn_block_scores(Q, K, 1, bs)
    kept = oracle.xattn_select(X, 0.6)
    rows = np.arange(L)
    got = oracle.attention_recall(Q, K, lambda h, r: oracle.xattn_row_mask(r, L, kept[h], bs), rows)
    want = np.mean([sum(X[h, I, kept[h][I]].sum() for I in range(L // bs)) / (L // bs) for h in range(2)])
    assert got == pytest.approx(want, rel=1e-12)
