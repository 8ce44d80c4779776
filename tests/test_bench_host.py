"""Host-side measurement code of bench.py: per-row active counts and the
per-worker work split of the striped / contiguous / ZigZag layouts."""
import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("L,bs,seed", [(512, 64, 0), (1024, 128, 1), (2048, 256, 2), (640, 64, 3)])
def test_row_counts_equal_explicit_mask(L, bs, seed):
    rng = np.random.default_rng(seed)
    nbs = L // bs
    V = np.sort(rng.choice(L, 25, replace=False))
    S = np.union1d(rng.choice(nbs, 3, replace=False), [0])
    counts = bench.row_active_counts(L, V, S, bs)
    assert np.array_equal(counts, oracle.explicit_mask(L, V, S, bs).sum(1))
    assert counts.sum() == oracle.active_entries(L, V, S, bs)


def test_shard_balance_dense_causal_closed_forms():
    """All bands kept (dense causal): row n has n + 1 entries, so ZigZag is
    exactly balanced, the contiguous split's heaviest worker is the last,
    and round-robin (striped) is balanced up to the first-row offset."""
    L, W = 8192, 8
    everything = [(np.array([], np.int64), np.arange(L // (64 * W)))]
    contig_all = [(np.array([], np.int64), np.arange(L // 64))]
    b = bench.shard_balance(L, W, everything, contig_all)
    assert b["zigzag_max_over_mean"] == 1.0
    C = L // W
    sums = np.array([C * C * r + C * (C + 1) // 2 for r in range(W)], np.float64)
    assert b["contiguous_max_over_mean"] == round(float(sums.max() / sums.mean()), 4)
    J = L // W
    st = np.array([sum(j * W + r + 1 for j in range(J)) for r in range(W)], np.float64)
    assert b["striped_max_over_mean"] == round(float(st.max() / st.mean()), 4)
    assert b["striped_total"] == b["contiguous_index_total"] == L * (L + 1) // 2
