"""Pins for the striped sparse ring attention oracle.

The ring runs W workers for W steps each, folding every step into a carried
(max, sum, output) state; the pages' striped layout makes the union of the
steps' local masks the global VS mask of the striped index (slash tiles of
64 W global tokens), so the ring must reproduce the single-pass masked
attention with ``stripes = W`` exactly (up to rounding), and every active
(query, key) pair must be visited by exactly one step.
"""
import numpy as np
import pytest

import oracle
from oracle.vs_oracle import _ring_step_mask


def _inputs(L, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    Q, K, V, dO = (rng.standard_normal((L, h, d)) for h in (Hq, Hkv, Hkv, Hq))
    K[[5, L // 3]] *= 4.0
    return Q, K, V, dO


def _index(L, W, Hq, seed):
    rng = np.random.default_rng(seed)
    nb = L // (64 * W)
    out = []
    for _ in range(Hq):
        S = np.union1d(rng.choice(nb, min(nb, 2), replace=False), [0])
        V = np.sort(rng.choice(L, 12, replace=False))
        out.append((V, S))
    return out


@pytest.mark.parametrize("L,W", [(512, 4), (2048, 32), (1024, 2)])
def test_steps_partition_the_global_mask(L, W):
    Vh, Sh = _index(L, W, 1, 1)[0]
    Ls = L // W
    glob = oracle.explicit_mask(L, Vh, Sh, 64 * W)
    cover = np.zeros((L, L), np.int64)
    for r in range(W):
        for t in range(W):
            s = (r - t) % W
            m = _ring_step_mask(Ls, W, r, s, Vh, Sh, 64)
            ii, jj = np.nonzero(m)
            np.add.at(cover, (ii * W + r, jj * W + s), 1)
    np.testing.assert_array_equal(cover, glob.astype(np.int64))


@pytest.mark.parametrize("L,W,Hq,Hkv", [(512, 4, 2, 1), (2048, 32, 2, 1), (1024, 2, 4, 2)])
def test_ring_equals_single_pass(L, W, Hq, Hkv):
    Q, K, V, dO = _inputs(L, Hq, Hkv, 16, L + W)
    index = _index(L, W, Hq, W)
    O, lse = oracle.striped_ring_forward(Q, K, V, index, W)
    Or, lser = oracle.attention_forward(Q, K, V, index, stripes=W)
    np.testing.assert_allclose(O, Or, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lser, rtol=1e-12, atol=1e-12)
    g = oracle.striped_ring_backward(Q, K, V, dO, index, W)
    gr = oracle.attention_backward(Q, K, V, dO, index, stripes=W)
    for a, b in zip(g, gr):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_step_with_empty_rows():
    # a worker's first local row at a step with s > r sees no key of that
    # shard (j < 0): its carried state stays empty and the merge skips it
    Vh, Sh = np.array([], np.int64), np.array([0])
    m = _ring_step_mask(64, 4, 0, 3, Vh, Sh, 64)
    assert not m[0].any() and m[1, 0] and not m[1, 1]
    m = _ring_step_mask(64, 4, 3, 0, Vh, Sh, 64)
    assert m[0, 0] and not m[0, 1]
