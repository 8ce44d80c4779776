"""Pins for the oracle's sparse-index approximation, mask and active count.

Definitions follow the MTraining review, section "分布式稀疏索引近似" (last_q
query rows scored against all keys, cumulative sums along vertical and slash
directions, the minimum number of lines that recall the target mass,
token-level verticals and 64x64 block slashes) and section "核心公式"
(sparsity ratio).  Each check below is independent of the oracle's own code:
brute force with explicit loops, exhaustive enumeration, conservation laws,
or a hand-worked fixture.
"""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import (active_entries, build_index, explicit_mask, index_scores,
                    select_budget, select_top_p, sparsity_ratio,
                    total_causal_entries)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_index_scores_brute_force_loops():
    L, Hq, Hkv, d, q = 48, 4, 2, 8, 5
    block, stripes = 4, 2
    Q, K = _rand((L, Hq, d), 1), _rand((L, Hkv, d), 2)
    v, S = index_scores(Q, K, q, stripes=stripes, block=block)
    bs = block * stripes
    scale = 1 / math.sqrt(d)
    for h in range(Hq):
        vb = [0.0] * L
        Sb = [0.0] * (L // bs)
        for i in range(q):
            n = L - q + i
            sc = [scale * sum(Q[n, h, c] * K[m, h // 2, c] for c in range(d)) for m in range(n + 1)]
            mx = max(sc)
            e = [math.exp(x - mx) for x in sc]
            tot = sum(e)
            for m in range(n + 1):
                vb[m] += e[m] / tot
                Sb[n // bs - m // bs] += e[m] / tot
        np.testing.assert_allclose(v[h], vb, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(S[h], Sb, rtol=1e-12, atol=1e-15)


def test_mass_conservation():
    L, Hq, d, q = 256, 3, 16, 64
    v, S = index_scores(_rand((L, Hq, d), 3), _rand((L, Hq, d), 4), q)
    np.testing.assert_allclose(v.sum(1), q, rtol=1e-12)
    np.testing.assert_allclose(S.sum(1), q, rtol=1e-12)
    assert (v >= 0).all() and (S >= 0).all()


def _min_k_exhaustive(x, p):
    tot = x.sum()
    for k in range(1, x.size + 1):
        best = max(sum(c) for c in itertools.combinations(x.tolist(), k))
        if best >= p * tot - 1e-15:
            return k
    return x.size


@pytest.mark.parametrize("seed", range(6))
def test_select_top_p_is_minimal_exhaustive(seed):
    rng = np.random.default_rng(seed)
    x = rng.exponential(size=10)
    if seed % 2:
        x[rng.integers(0, 10, 3)] = x[0]          # plant ties
    for p in (0.3, 0.5, 0.9, 0.99):
        sel = select_top_p(x, p)
        assert len(sel) == _min_k_exhaustive(x, p)
        assert x[sel].sum() >= p * x.sum() * (1 - 1e-15)
        # the kept set is a top set: nothing outside beats anything inside,
        # and among equal values the lower index is kept
        out = np.setdiff1d(np.arange(x.size), sel)
        if out.size:
            assert x[sel].min() >= x[out].max()
            thr = x[sel].min()
            tied_out = out[x[out] == thr]
            tied_in = sel[x[sel] == thr]
            if tied_out.size:
                assert tied_in.max() < tied_out.min()
        # dropping the smallest kept element leaves less than p
        if sel.size > 1:
            assert x[sel].sum() - x[sel].min() < p * x.sum()


def test_select_top_p_one_keeps_all_positive():
    x = np.array([0.5, 0.0, 1e-300, 2.0, 0.0])
    np.testing.assert_array_equal(select_top_p(x, 1.0), [0, 2, 3])


def test_planted_outlier_becomes_vertical():
    # a key aligned with the last queries' mean direction, scaled x8, must be
    # kept as a vertical (outlier keys => vertical lines)
    L, d, q = 512, 64, 64
    rng = np.random.default_rng(7)
    Q = rng.standard_normal((L, 1, d))
    K = rng.standard_normal((L, 1, d))
    pos = [37, 200, 311]
    u = Q[L - q:, 0].mean(0)
    u /= np.linalg.norm(u)
    for m in pos:
        K[m, 0] = 8.0 * math.sqrt(d) * u
    index, v, S = build_index(Q, K, q, 0.9)
    Vh, Sh = index[0]
    assert set(pos) <= set(Vh.tolist())
    assert 0 in Sh.tolist()


def _read_golden(name):
    rec = {"mask": []}
    for line in open(os.path.join(GOLDEN, name)):
        if not line.strip() or line.startswith("#"):
            continue
        k, *vals = line.split()
        if k == "mask":
            rec["mask"].append([int(c) for c in vals[0]])
        else:
            rec[k] = [int(x) for x in vals]
    return rec


def test_hand_worked_mask_fixture():
    g = _read_golden("vs_mask_L8_bs2.txt")
    L, bs = g["L"][0], g["bs"][0]
    msk = explicit_mask(L, np.array(g["V"]), np.array(g["S"]), bs)
    np.testing.assert_array_equal(msk.astype(int), np.array(g["mask"]))
    assert active_entries(L, np.array(g["V"]), np.array(g["S"]), bs) == g["active"][0]
    assert total_causal_entries(L) == g["total"][0]
    assert abs(sparsity_ratio(L, 1, g["active"][0]) - (1 - 24 / 36)) < 1e-15


@pytest.mark.parametrize("seed", range(8))
def test_active_entries_equals_mask_count(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4, 8]))
    nbs = int(rng.integers(1, 12))
    L = bs * nbs
    S = np.union1d(rng.choice(nbs, rng.integers(0, nbs + 1), replace=False), [0])
    V = np.sort(rng.choice(L, rng.integers(0, L + 1), replace=False))
    msk = explicit_mask(L, V, S, bs)
    assert active_entries(L, V, S, bs) == int(msk.sum())
    # every row keeps at least its diagonal entry
    assert msk[np.arange(L), np.arange(L)].all()


def test_striped_local_tiles_are_global_tiles():
    """Striped layout (round-robin tokens over W workers): token t lives on
    shard t % W at local position t // W.  A slash band measured in 64-wide
    tiles of local positions and the local causal rule (key j allowed for
    query i iff j <= i when its shard s <= r, else j < i) give the same mask
    as global tiles of 64 * W tokens, which is what the oracle uses."""
    W, block, nloc = 4, 2, 6            # L = 24, global tiles of 8 tokens
    L = W * block * nloc
    rng = np.random.default_rng(5)
    S = np.union1d(rng.choice(nloc, 3, replace=False), [0])
    V = np.sort(rng.choice(L, 5, replace=False))
    ref = np.zeros((L, L), bool)
    for n in range(L):
        r, i = n % W, n // W
        for m in range(L):
            s, j = m % W, m // W
            causal = (j <= i) if s <= r else (j < i)
            if causal and ((i // block - j // block) in set(S.tolist()) or m in set(V.tolist())):
                ref[n, m] = True
    np.testing.assert_array_equal(explicit_mask(L, V, S, block * W), ref)


@pytest.mark.parametrize("seed", range(5))
def test_budget_fill_brute_force(seed):
    rng = np.random.default_rng(seed)
    bs, nbs = 4, 6
    L = bs * nbs
    v = rng.exponential(size=L) * (rng.random(L) < 0.7)
    S = rng.exponential(size=nbs) * 3
    if seed == 3:
        v[5] = S[2]                     # a vertical/slash tie
    T = total_causal_entries(L)
    for dens in (0.05, 0.3, 0.6, 0.95):
        Vs, Ss = select_budget(v, S, L, bs, dens)
        # brute force over every candidate threshold, mask counted explicitly
        cands = sorted(set([x for x in np.concatenate([S[1:], v]) if x > 0]), reverse=True)
        best = None
        base = explicit_mask(L, [], [0], bs).sum()
        if base >= dens * T:
            best = ([], [0])
        else:
            for tau in cands:
                Vt = [m for m in range(L) if v[m] >= tau]
                St = [0] + [B for B in range(1, nbs) if S[B] >= tau]
                if explicit_mask(L, Vt, St, bs).sum() >= dens * T:
                    best = (Vt, St)
                    break
            if best is None:
                tau = cands[-1]
                best = ([m for m in range(L) if v[m] >= tau], [0] + [B for B in range(1, nbs) if S[B] >= tau])
        np.testing.assert_array_equal(Vs, best[0])
        np.testing.assert_array_equal(Ss, best[1])


def test_build_index_recall_at_least_p():
    L, Hq, Hkv, d, q = 1024, 4, 2, 32, 64
    rng = np.random.default_rng(11)
    Q, K = rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d))
    K[rng.choice(L, 4, replace=False)] *= 6
    for p in (0.5, 0.9):
        index, v, S = build_index(Q, K, q, p)
        for h, (Vh, Sh) in enumerate(index):
            assert v[h, Vh].sum() >= p * v[h].sum() * (1 - 1e-14)
            assert S[h, Sh].sum() >= p * S[h].sum() * (1 - 1e-14)
            assert np.all(np.diff(Vh) > 0) and np.all(np.diff(Sh) > 0) and Sh[0] == 0


def test_group_shared_index_is_the_union_of_masks():
    """Brute force: each head's mask under the group-shared index is the OR of
    the explicit masks of its group's per-head indices, the exact active
    count equals the mask's, and every head's vertical recall is at least
    that of its own selection."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(4)
    L, G, Hkv, bs = 256, 4, 2, 64
    nb = L // bs
    per_head = [(np.sort(rng.choice(L, rng.integers(0, 9), replace=False)),
                 np.union1d(rng.choice(nb, rng.integers(0, 3), replace=False), [0])) for _ in range(G * Hkv)]
    shared = oracle.group_shared_index(per_head, G)
    for h in range(G * Hkv):
        g = h // G
        want = np.zeros((L, L), bool)
        for hh in range(g * G, (g + 1) * G):
            want |= oracle.explicit_mask(L, *per_head[hh], bs)
        got = oracle.explicit_mask(L, *shared[h], bs)
        assert (got == want).all()
        assert oracle.active_entries(L, *shared[h], bs) == int(want.sum())
        assert set(per_head[h][0].tolist()) <= set(shared[h][0].tolist())
        assert set(per_head[h][1].tolist()) <= set(shared[h][1].tolist())


def test_build_index_group_mode():
    import numpy as np
    import oracle
    rng = np.random.default_rng(8)
    L, Hq, Hkv, d = 512, 4, 2, 16
    Q, K = rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d))
    K[[10, 300]] *= 5
    per, v, S = oracle.build_index(Q, K, 32, 0.9)
    grp, v2, S2 = oracle.build_index(Q, K, 32, 0.9, index_mode=1)
    assert np.array_equal(v, v2) and np.array_equal(S, S2)
    for h in range(Hq):
        ref = oracle.group_shared_index(per, Hq // Hkv)[h]
        assert np.array_equal(grp[h][0], ref[0]) and np.array_equal(grp[h][1], ref[1])
        # recall of every head's own mass stays >= top_p under the union
        assert v[h][grp[h][0]].sum() >= 0.9 * v[h].sum() - 1e-12
        assert S[h][grp[h][1]].sum() >= 0.9 * S[h].sum() - 1e-12
