"""Pins for the oracle's masked attention forward and backward.

Checks against (1) PyTorch's dense scaled-dot-product attention in fp64 on
the CPU when every line is kept (the VS mask then equals the causal mask),
(2) PyTorch autograd through an explicitly masked softmax, (3) central finite
differences, and (4) explicit per-entry loops.  The online softmax across KV
blocks in the ring-attention page (section 2.1) computes exactly this
masked softmax, so the oracle is the definition itself.
"""
import math

import numpy as np
import pytest
import torch

from oracle import (attention_backward, attention_forward, attention_forward_rows,
                    explicit_mask)


def _inputs(L, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d)),
            rng.standard_normal((L, Hkv, d)), rng.standard_normal((L, Hq, d)))


def _torch_masked(Q, K, V, masks, dO):
    Hq, G = Q.shape[1], Q.shape[1] // K.shape[1]
    q = torch.tensor(Q, dtype=torch.float64).permute(1, 0, 2).requires_grad_()
    k = torch.tensor(K, dtype=torch.float64).permute(1, 0, 2).requires_grad_()
    v = torch.tensor(V, dtype=torch.float64).permute(1, 0, 2).requires_grad_()
    ke, ve = k.repeat_interleave(G, 0), v.repeat_interleave(G, 0)
    m = torch.tensor(np.stack(masks))
    o = torch.nn.functional.scaled_dot_product_attention(q, ke, ve, attn_mask=m)
    o.backward(torch.tensor(dO, dtype=torch.float64).permute(1, 0, 2))
    return (o.detach().permute(1, 0, 2).numpy(), q.grad.permute(1, 0, 2).numpy(),
            k.grad.permute(1, 0, 2).numpy(), v.grad.permute(1, 0, 2).numpy())


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (4, 1)])
def test_all_lines_kept_equals_dense_causal(Hq, Hkv):
    L, d, bs = 256, 16, 64
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, Hq * 10 + Hkv)
    index = [(np.array([], np.int64), np.arange(L // bs))] * Hq
    O, LSE = attention_forward(Q, K, V, index)
    G = Hq // Hkv
    q = torch.tensor(Q).permute(1, 0, 2)
    k = torch.tensor(K).permute(1, 0, 2).repeat_interleave(G, 0)
    v = torch.tensor(V).permute(1, 0, 2).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(O, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    s = (q @ k.transpose(1, 2)) / math.sqrt(d)
    s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12)
    # all verticals kept, only band 0: also dense causal
    index2 = [(np.arange(L), np.array([0]))] * Hq
    O2, _ = attention_forward(Q, K, V, index2)
    np.testing.assert_allclose(O2, O, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_masked_fwd_bwd_vs_autograd(seed):
    L, Hq, Hkv, d, bs = 128, 4, 2, 8, 16
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 100 + seed)
    rng = np.random.default_rng(seed)
    index, masks = [], []
    for h in range(Hq):
        S = np.union1d(rng.choice(L // bs, 3, replace=False), [0])
        Vv = np.sort(rng.choice(L, 9, replace=False))
        index.append((Vv, S))
        masks.append(explicit_mask(L, Vv, S, bs))
    O, _ = attention_forward(Q, K, V, index, block=bs)
    dQ, dK, dV = attention_backward(Q, K, V, dO, index, block=bs)
    rO, rdQ, rdK, rdV = _torch_masked(Q, K, V, masks, dO)
    for a, b in ((O, rO), (dQ, rdQ), (dK, rdK), (dV, rdV)):
        np.testing.assert_allclose(a, b, atol=1e-11, rtol=1e-11)


def test_backward_finite_differences():
    L, Hq, Hkv, d, bs = 16, 2, 1, 4, 4
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 9)
    index = [(np.array([1, 6]), np.array([0, 2])), (np.array([0]), np.array([0, 1, 3]))]
    dQ, dK, dV = attention_backward(Q, K, V, dO, index, block=bs)

    def f(Qx, Kx, Vx):
        O, _ = attention_forward(Qx, Kx, Vx, index, block=bs)
        return float((O * dO).sum())

    eps = 1e-6
    rng = np.random.default_rng(0)
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        for _ in range(12):
            idx = tuple(rng.integers(0, s) for s in X.shape)
            old = X[idx]
            X[idx] = old + eps
            fp = f(Q, K, V)
            X[idx] = old - eps
            fm = f(Q, K, V)
            X[idx] = old
            num = (fp - fm) / (2 * eps)
            assert abs(num - G[idx]) <= 1e-7 * max(1.0, abs(G[idx]))


def test_forward_explicit_loops():
    L, d, bs = 40, 3, 4
    Q, K, V, _ = _inputs(L, 1, 1, d, 21)
    Vv, S = np.array([2, 13, 30]), np.array([0, 3, 5])
    O, LSE = attention_forward(Q, K, V, [(Vv, S)], block=bs)
    for n in range(L):
        act = [m for m in range(n + 1)
               if (n // bs - m // bs) in (0, 3, 5) or m in (2, 13, 30)]
        sc = [sum(Q[n, 0, c] * K[m, 0, c] for c in range(d)) / math.sqrt(d) for m in act]
        mx = max(sc)
        e = [math.exp(x - mx) for x in sc]
        for c in range(d):
            ref = sum(e[j] * V[act[j], 0, c] for j in range(len(act))) / sum(e)
            assert abs(O[n, 0, c] - ref) < 1e-12
        assert abs(LSE[0, n] - (mx + math.log(sum(e)))) < 1e-12


def test_rows_subset_matches_full():
    L, Hq, Hkv, d = 192, 2, 1, 8
    Q, K, V, _ = _inputs(L, Hq, Hkv, d, 5)
    index = [(np.array([3, 70]), np.array([0, 1])), (np.array([], np.int64), np.array([0, 2]))]
    O, LSE = attention_forward(Q, K, V, index)
    rows = np.array([0, 63, 64, 191, 100])
    Or, LSEr = attention_forward_rows(Q, K, V, index, rows)
    np.testing.assert_allclose(Or, O[rows], atol=1e-14)
    np.testing.assert_allclose(LSEr, LSE[:, rows], atol=1e-14)


def test_dq_rows_matches_full_backward():
    from oracle import attention_backward_dq_rows
    L, Hq, Hkv, d = 256, 4, 2, 8
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 31)
    rng = np.random.default_rng(4)
    index = [(np.sort(rng.choice(L, 7, replace=False)), np.union1d(rng.choice(4, 2, replace=False), [0]))
             for _ in range(Hq)]
    dQ, _, _ = attention_backward(Q, K, V, dO, index)
    rows = np.array([0, 5, 64, 200, 255])
    np.testing.assert_allclose(attention_backward_dq_rows(Q, K, V, dO, index, rows), dQ[rows], atol=1e-13)


@pytest.mark.parametrize("stripes", [1, 2])
def test_dkdv_keys_matches_full_backward(stripes):
    """dK / dV of listed keys against the full backward: keys in the first,
    a middle and the last tile, kept verticals among them (rows from the
    vertical on), GQA 4 / 2, and the striped tiles."""
    from oracle import attention_backward_dkdv_keys
    L, Hq, Hkv, d = 512, 4, 2, 8
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 41 + stripes)
    rng = np.random.default_rng(6)
    nbs = L // (64 * stripes)
    index = [(np.sort(np.union1d(rng.choice(L, 9, replace=False), [200])),
              np.union1d(rng.choice(nbs, 2, replace=False), [0])) for _ in range(Hq)]
    _, dK, dV = attention_backward(Q, K, V, dO, index, stripes=stripes)
    verts = np.unique(np.concatenate([V_ for V_, _ in index]))
    plain = np.setdiff1d([0, 3, 63, 201, 330, 448, 500, 511], verts)
    # keys that are no head's vertical (rows only from the kept bands), then
    # with two verticals among them (rows from the earlier one on)
    assert verts[0] < 200
    for keys in (plain, np.union1d(plain, [verts[0], 200])):
        gK, gV = attention_backward_dkdv_keys(Q, K, V, dO, index, keys, stripes=stripes)
        np.testing.assert_allclose(gK, dK[keys], atol=1e-13)
        np.testing.assert_allclose(gV, dV[keys], atol=1e-13)


def test_gradient_column_identities():
    """Identities used for full-size checks: summed over keys, dV equals the
    sum of dO over the rows of the group's heads (softmax rows sum to 1), and
    dK sums to zero (each row of dS sums to zero)."""
    L, Hq, Hkv, d = 128, 4, 2, 8
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 32)
    rng = np.random.default_rng(5)
    index = [(np.sort(rng.choice(L, 5, replace=False)), np.array([0, 1])) for _ in range(Hq)]
    _, dK, dV = attention_backward(Q, K, V, dO, index)
    for g in range(Hkv):
        np.testing.assert_allclose(dV[:, g].sum(0), dO[:, g * 2:(g + 1) * 2].sum((0, 1)), atol=1e-10)
        np.testing.assert_allclose(dK[:, g].sum(0), 0.0, atol=1e-10)


def test_bf16_round_known_values():
    from oracle import bf16_round
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: the even significand (1) wins;
    # 1 + 3 * 2^-8 ties up to 1 + 2^-6 (even); 1 + 2^-20 rounds down; 3e38
    # rounds to the bf16 pattern 0x7F62 (fp32 first, then bf16, both RNE)
    x = np.array([1.0, 1.00390625, 1.01171875, 1.0078125, -2.5, 1.0 + 2.0 ** -20, 0.0, 3.0e38])
    big = float(np.array([0x7F62 << 16], np.uint32).view(np.float32)[0])
    np.testing.assert_array_equal(bf16_round(x), [1.0, 1.0, 1.015625, 1.0078125, -2.5, 1.0, 0.0, big])


def _explicit_bf16_backward(Q, K, V, dO, masks, scale):
    """Per-entry loops: the stated roundings applied element by element."""
    from oracle import bf16_round
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    r = lambda x: float(bf16_round(np.array([x]))[0])
    for h in range(Hq):
        g = h // G
        for n in range(L):
            act = [m for m in range(L) if masks[h][n, m]]
            s = {m: scale * sum(Q[n, h, c] * K[m, g, c] for c in range(d)) for m in act}
            mx = max(s.values())
            z = sum(math.exp(s[m] - mx) for m in act)
            P = {m: math.exp(s[m] - mx) / z for m in act}
            O = [r(sum(P[m] * V[m, g, c] for m in act)) for c in range(d)]
            D = sum(dO[n, h, c] * O[c] for c in range(d))
            for m in act:
                dP = sum(dO[n, h, c] * V[m, g, c] for c in range(d))
                dS = r(P[m] * (dP - D))
                pb = r(P[m])
                for c in range(d):
                    dV[m, g, c] += pb * dO[n, h, c]
                    dQ[n, h, c] += scale * dS * K[m, g, c]
                    dK[m, g, c] += scale * dS * Q[n, h, c]
    return dQ, dK, dV


def test_bf16_products_backward_explicit_loops():
    from oracle import attention_backward_bf16_products
    L, Hq, Hkv, d = 40, 2, 1, 8
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 11)
    index = [(np.array([3, 17, 30]), np.array([0, 2])), (np.array([1, 8]), np.array([0, 1, 3]))]
    masks = [explicit_mask(L, Vh, Sh, 8) for Vh, Sh in index]
    scale = 1.0 / math.sqrt(d)
    ref = _explicit_bf16_backward(Q, K, V, dO, masks, scale)
    got = attention_backward_bf16_products(Q, K, V, dO, index, block=8)
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g, e, rtol=1e-12, atol=1e-12)


def test_bf16_products_backward_within_first_order_bound():
    """|emulated - exact| is bounded entry by entry by the unit roundoff
    u = 2^-8 times the magnitudes the three roundings touch: dV by
    u sum_n P |dO|; dQ and dK by scale sum (u |dS'| + P u sum_c |dO O|) |k|
    (resp. |q|), with dS' = P (dP - D) formed from the rounded O."""
    from oracle import attention_backward_bf16_products, bf16_round
    L, Hq, Hkv, d = 96, 2, 1, 16
    Q, K, V, dO = _inputs(L, Hq, Hkv, d, 5)
    K[[7, 50]] *= 6.0
    index = [(np.array([7, 50, 71]), np.array([0, 1, 4])), (np.array([7, 50]), np.array([0, 2]))]
    u = 2.0 ** -8
    scale = 1.0 / math.sqrt(d)
    exact = attention_backward(Q, K, V, dO, index, block=16)
    emu = attention_backward_bf16_products(Q, K, V, dO, index, block=16)
    bQ, bK, bV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for h, (Vh, Sh) in enumerate(index):
        m = explicit_mask(L, Vh, Sh, 16)
        s = np.where(m, scale * Q[:, h] @ K[:, 0].T, -np.inf)
        P = np.exp(s - s.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        O = P @ V[:, 0]
        Ob = bf16_round(O)
        dSp = P * (dO[:, h] @ V[:, 0].T - (dO[:, h] * Ob).sum(1, keepdims=True))
        w = u * np.abs(dSp) + P * u * (np.abs(dO[:, h]) * np.abs(O)).sum(1, keepdims=True)
        bV[:, 0] += u * P.T @ np.abs(dO[:, h])
        bQ[:, h] = scale * w @ np.abs(K[:, 0])
        bK[:, 0] += scale * w.T @ np.abs(Q[:, h])
    for e, x, b in zip(emu, exact, (bQ, bK, bV)):
        assert (np.abs(e - x) <= b * (1 + 1e-6) + 1e-12).all()
        assert np.abs(e - x).max() > 0      # the roundings do happen
