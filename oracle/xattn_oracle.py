"""Plain fp64 CPU oracle for the anti-diagonal block scorer (an alternative
sparse index, the ablation row "MTraining w/ XAttn Idx.").

TEST INFRASTRUCTURE ONLY, like ``vs_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may run
it.  It shares no code with the CUDA library.

Source: the MTraining paper review ("MTraining: 分布式动态稀疏注意力高效超长
上下文训练"), section 五 "实验结果", table "训练效率结果" (the ablation row
that replaces the VS index by an XAttention index), and section 七 "技术影响",
table "与现有方法对比" (XAttention: efficient at inference, its anti-slash
pattern does not match ring attention).  The pages name the scorer and
nothing more.  The reading taken here is the published XAttention block
scorer, restated:

* Strided cells: with stride S, query group r holds tokens rS .. rS+S-1 and
  key group c tokens cS .. cS+S-1.  Cell (r, c) is scored by the mean of the
  S scaled logits on the anti-diagonal of that S x S sub-block, the entries
  (rS + j, cS + S-1-j), j = 0 .. S-1:
      z[r, c] = scale / S * sum_j q[rS + j] . k[cS + S-1-j].
* Causality at cell granularity: cells with c <= r are kept (the diagonal
  cell included, as its anti-diagonal starts below the diagonal), cells with
  c > r are masked.
* P = softmax over the kept cells of each strided row.
* Block score of block row I and block column J (blocks of bs tokens, bs/S
  strided rows and columns each): the mass of the cells of (I, J) averaged
  over the block's bs/S strided rows, so every block row sums to one:
      X[I, J] = (S / bs) * sum_{r in I, c in J} P[r, c].
* Selection per block row I (the method's top-p rule applied to blocks):
  the smallest descending prefix of X[I, 0..I] (ties: lower J first) whose
  sum reaches ``threshold`` of the row's total, plus the diagonal block I,
  which is always kept.  threshold >= 1 keeps every block of positive score.
* Stripes: the block edge is bs = 64 * W, the same tiles the VS path uses
  for the striped layout (64 x 64 shard-local tiles are global bs x bs
  tiles).
* GQA: query head h scores against key/value head h // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np

from .vs_oracle import select_top_p

__all__ = ["xattn_block_scores", "xattn_select", "xattn_active_entries", "xattn_row_mask",
           "attention_recall"]


def xattn_block_scores(Q, K, stride: int, bs: int, scale: float | None = None, block_rows=None):
    """Block scores X [Hq, nI, nb] (fp64) for the listed block rows (all rows
    when ``block_rows`` is None; then X is [Hq, nb, nb] with zeros above the
    diagonal).  Q [L, Hq, d], K [L, Hkv, d]; L a multiple of bs, bs of the
    stride."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    S = int(stride)
    R, nb, bsS = L // S, L // bs, bs // S
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows_I = np.arange(nb) if block_rows is None else np.asarray(block_rows, np.int64)
    X = np.zeros((Hq, rows_I.size, nb))
    c = np.arange(R)
    for h in range(Hq):
        # ks[c, j] = k[cS + S-1-j]: the key of the anti-diagonal entry in row j
        ks = K[:, h // G, :].reshape(R, S, d)[:, ::-1, :]
        for n, I in enumerate(rows_I.tolist()):
            r = np.arange(I * bsS, (I + 1) * bsS)
            qs = Q[I * bs:(I + 1) * bs, h, :].reshape(bsS, S, d)  # qs[r, j] = q[rS + j]
            z = np.einsum("rjx,cjx->rc", qs, ks) * (scale / S)
            z = np.where(c[None, :] <= r[:, None], z, -np.inf)
            z = z - z.max(axis=1, keepdims=True)
            P = np.exp(z)
            P /= P.sum(axis=1, keepdims=True)
            X[h, n] = P.reshape(bsS, nb, bsS).sum(axis=(0, 2)) / bsS
    return X


def xattn_select(X, threshold: float, block_rows=None):
    """Kept block columns per head and block row: a list over heads of lists
    over the block rows of ascending int64 arrays.  X as returned by
    ``xattn_block_scores`` (block row n of X is block row block_rows[n])."""
    X = np.asarray(X, np.float64)
    Hq, nI, nb = X.shape
    rows_I = np.arange(nb) if block_rows is None else np.asarray(block_rows, np.int64)
    out = []
    for h in range(Hq):
        kept = []
        for n, I in enumerate(rows_I.tolist()):
            sel = select_top_p(X[h, n, :I + 1], threshold)
            kept.append(np.union1d(sel, [I]).astype(np.int64))
        out.append(kept)
    return out


def xattn_active_entries(kept_rows, bs: int) -> int:
    """Causal entries inside the kept blocks of one head: bs * bs per kept
    block below the diagonal, bs (bs + 1) / 2 for the diagonal block."""
    A = 0
    for I, J in enumerate(kept_rows):
        J = np.asarray(J, np.int64)
        A += int((J < I).sum()) * bs * bs + int((J == I).sum()) * (bs * (bs + 1) // 2)
    return A


def xattn_row_mask(rows: np.ndarray, L: int, kept_rows, bs: int) -> np.ndarray:
    """Boolean [len(rows), L] mask of token rows under one head's block index:
    entry (n, m) is active iff m <= n and block (n // bs, m // bs) is kept."""
    rows = np.asarray(rows, np.int64)
    nb = L // bs
    keep = np.zeros((nb, nb), bool)
    for I, J in enumerate(kept_rows):
        keep[I, np.asarray(J, np.int64)] = True
    m = np.arange(L)
    return (m[None, :] <= rows[:, None]) & keep[(rows // bs)[:, None], (m // bs)[None, :]]


def attention_recall(Q, K, mask_fn, rows, scale: float | None = None) -> float:
    """Mean over heads and the listed query rows of the exact causal
    attention mass (fp64 softmax of scale q.k over m <= n) that falls on the
    active entries of ``mask_fn(h, rows)`` (boolean [len(rows), L])."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.asarray(rows, np.int64)
    m = np.arange(L)
    tot = 0.0
    for h in range(Hq):
        s = scale * (Q[rows, h, :] @ K[:, h // G, :].T)
        s = np.where(m[None, :] <= rows[:, None], s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        tot += float((p * mask_fn(h, rows)).sum())
    return tot / (Hq * rows.size)
