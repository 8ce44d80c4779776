"""Plain fp64 CPU oracle for dynamic vertical-slash (VS) sparse causal attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in ``oracle/``.
It shares no code with the CUDA library and never imports it.

Sources (web pages on the method; cited by page title and section):

* [MT] "MTraining: 分布式动态稀疏注意力高效超长上下文训练" (paper review of
  MTraining, arXiv 2510.18830).  Sections used: 三/核心创新/1 "Vertical-Slash
  稀疏模式" (the VS pattern and the RoPE expectation equation), 三/核心创新/2
  "分布式稀疏索引近似" (last_q scoring, vertical and slash cumulative sums,
  minimum set of lines recalling the target mass, token-level verticals and
  64x64 block-level slashes, active-region derivation), 三/核心创新/3 "平衡稀疏
  环注意力" (striped layout), 四 "核心公式" (sparsity ratio), 五/训练损失分析
  ("online top-p budget"), 五/实验设置 (YaRN factor 32), 八/局限性 4 (sparsity
  fixed at 95 % in the experiments).
* [RA] "Ring Attention：突破长序列训练的分布式架构", §2.1 (incremental softmax
  over KV blocks) and §3.1 (striped round-robin layout).

Everything is fp64.  Readings of points the pages leave open (each is listed
in the design notes with its justification):

* softmax scale 1/sqrt(d) in the index and in attention;
* index scores are per-row softmax probabilities of the last ``last_q`` query
  rows, so each row carries mass 1 and each direction's total mass is last_q;
* vertical and slash budgets are chosen independently, each the smallest
  prefix of the descending order (ties: lower index first) whose cumulative
  mass reaches ``top_p`` of the total; ``top_p == 1`` keeps every positive one;
* slash band ``B`` of a (query n, key m) pair is ``n//bs - m//bs`` with
  ``bs = 64 * stripes`` (64x64 tiles in shard-local coordinates of the striped
  layout are exactly global ``bs x bs`` tiles); band 0 is always kept;
* entry (n, m) is active iff ``m <= n`` and (its band is kept or ``m`` is a
  kept vertical);
* GQA: every query head has its own index; key/value head = h // (Hq // Hkv).

Parity unpinned: YaRN's NTK-by-parts frequencies (the pages only name the
method and its factor); see ``rope_inv_freq``.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_round", "rope_inv_freq", "rope_mscale", "rope", "index_scores",
    "select_top_p", "select_budget", "build_index", "active_entries",
    "sparsity_ratio", "explicit_mask", "attention_forward", "attention_backward",
    "attention_forward_rows", "attention_backward_dq_rows", "attention_backward_dkdv_keys",
    "total_causal_entries",
    "attention_backward_bf16_products", "striped_ring_forward", "striped_ring_backward",
    "group_shared_index",
]


# ----------------------------------------------------------------------------
# small helpers

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (through fp32, round-to-nearest-even at each
    step) and return them as fp64.  Used where the oracle itself must hand a
    bf16 tensor to the next step (e.g. RoPE output stored as bf16)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def total_causal_entries(L: int) -> int:
    """Entries of one head's causal attention matrix: L (L + 1) / 2."""
    return L * (L + 1) // 2


# ----------------------------------------------------------------------------
# RoPE  ([MT] 三/核心创新/1: the expectation equation fixes the rotate-half
# convention: channel i pairs with i + d/2, theta_i = base^(-2i/d))

def rope_inv_freq(d: int, theta: float, yarn_factor: float = 1.0,
                  yarn_orig_len: int = 0, beta_fast: float = 32.0,
                  beta_slow: float = 1.0) -> np.ndarray:
    """Per-pair angular frequency theta_i = theta^(-2i/d), i < d/2.

    With ``yarn_factor`` s > 1 the frequencies follow YaRN's NTK-by-parts
    interpolation (Peng et al. 2024; the pages only name "YaRN, factor 32"):
    r_i = orig_len * theta_i / (2 pi) full turns over the original context,
    gamma_i = clip((r_i - beta_slow) / (beta_fast - beta_slow), 0, 1),
    theta'_i = theta_i * (gamma_i + (1 - gamma_i) / s).  (Parity unpinned
    beyond its limiting cases.)"""
    i = np.arange(d // 2, dtype=np.float64)
    f = theta ** (-2.0 * i / d)
    if yarn_factor > 1.0:
        r = yarn_orig_len * f / (2.0 * math.pi)
        g = np.clip((r - beta_slow) / (beta_fast - beta_slow), 0.0, 1.0)
        f = f * (g + (1.0 - g) / yarn_factor)
    return f


def rope_mscale(yarn_factor: float) -> float:
    """YaRN attention temperature folded into q and k: 0.1 ln s + 1 (s > 1)."""
    return 0.1 * math.log(yarn_factor) + 1.0 if yarn_factor > 1.0 else 1.0


def rope(x: np.ndarray, theta: float, positions: np.ndarray | None = None,
         transpose: bool = False, yarn_factor: float = 1.0,
         yarn_orig_len: int = 0) -> np.ndarray:
    """Rotate-half RoPE of ``x`` [L, H, d] at token positions ``positions``.

    For i < d/2 with phi = t * theta_i:
      y_i       = c * (x_i cos phi - x_{i+d/2} sin phi)
      y_{i+d/2} = c * (x_{i+d/2} cos phi + x_i sin phi)
    where c is the YaRN temperature (1 without YaRN).  ``transpose=True``
    applies the adjoint c * R(phi)^T (rotation by -phi), which maps gradients
    of the rotated tensor back to the un-rotated one."""
    x = np.asarray(x, dtype=np.float64)
    L, H, d = x.shape
    t = np.arange(L, dtype=np.float64) if positions is None else np.asarray(positions, np.float64)
    f = rope_inv_freq(d, theta, yarn_factor, yarn_orig_len)
    phi = t[:, None] * f[None, :]                     # [L, d/2]
    c, s = np.cos(phi)[:, None, :], np.sin(phi)[:, None, :]
    if transpose:
        s = -s
    a, b = x[..., : d // 2], x[..., d // 2:]
    y = np.empty_like(x)
    y[..., : d // 2] = a * c - b * s
    y[..., d // 2:] = b * c + a * s
    return y * rope_mscale(yarn_factor)


# ----------------------------------------------------------------------------
# Sparse-index approximation ([MT] 三/核心创新/2)

def index_scores(Q: np.ndarray, K: np.ndarray, last_q: int, scale: float | None = None,
                 stripes: int = 1, block: int = 64):
    """Vertical and slash attention mass of the last ``last_q`` query rows.

    Rows n_i = L - last_q + i.  s_{i,m} = scale * q_{n_i} . k_m for m <= n_i,
    p_{i,m} = softmax over m.  Returns
      v [Hq, L]   v[h, m] = sum_i p_{i,m}                       (vertical lines)
      S [Hq, L/bs] S[h, B] = sum of p_{i,m} over n_i//bs - m//bs == B  (slash bands)
    with bs = block * stripes."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    L, Hq, d = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    nbs = L // bs
    n = np.arange(L - last_q, L)
    m = np.arange(L)
    causal = m[None, :] <= n[:, None]
    band = (n // bs)[:, None] - (m // bs)[None, :]
    v = np.zeros((Hq, L))
    S = np.zeros((Hq, nbs))
    for h in range(Hq):
        s = scale * (Q[n, h, :] @ K[:, h // G, :].T)
        s = np.where(causal, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        v[h] = p.sum(axis=0)
        S[h] = np.bincount(band[causal], weights=p[causal], minlength=nbs)[:nbs]
    return v, S


def select_top_p(x: np.ndarray, p: float) -> np.ndarray:
    """Smallest prefix of ``x`` sorted descending (ties: lower index first)
    whose cumulative sum reaches ``p`` of the total; returned as ascending
    indices.  ``p >= 1`` keeps every positive element ("minimum number of
    lines that recall the target mass", [MT] 三/核心创新/2)."""
    x = np.asarray(x, np.float64)
    if p >= 1.0:
        return np.flatnonzero(x > 0).astype(np.int64)
    order = np.argsort(-x, kind="stable")
    c = np.cumsum(x[order])
    k = int(np.searchsorted(c, p * c[-1], side="left")) + 1
    return np.sort(order[:min(k, x.size)]).astype(np.int64)


def active_entries(L: int, V: np.ndarray, S: np.ndarray, bs: int = 64) -> int:
    """Exact number of active (n, m) entries of one head's VS mask.

    Kept band B >= 1 covers (L/bs - B) full bs x bs tiles; band 0 covers the
    causal halves of the diagonal tiles; a kept vertical m adds bs entries
    for every later row tile r whose band r - m//bs is not kept (its own
    tile is inside band 0, earlier tiles are above the diagonal)."""
    nbs = L // bs
    S = np.asarray(S, np.int64)
    V = np.asarray(V, np.int64)
    inS = np.zeros(nbs, bool)
    inS[S] = True
    A = 0
    for B in S.tolist():
        A += nbs * (bs * (bs + 1) // 2) if B == 0 else (nbs - B) * bs * bs
    # notS[x] = #{B in [1, x] : B not kept}
    notS = np.concatenate([[0], np.cumsum(~inS[1:])])
    for mm in V.tolist():
        A += bs * int(notS[nbs - 1 - mm // bs])
    return int(A)


def sparsity_ratio(L: int, Hq: int, A_total: int) -> float:
    """1 - active entries / total causal entries ([MT] 四 核心公式)."""
    return 1.0 - A_total / (Hq * total_causal_entries(L))


def select_budget(v: np.ndarray, S: np.ndarray, L: int, bs: int, density: float):
    """Budget-fill selection at a fixed active density.

    The pages' experiments fix the sparsity at 95 % ([MT] 八/4) while the
    method selects by top-p; this variant reaches a given density with the
    same scores.  Verticals (v[m]) and slash bands B >= 1 (S[B]) are ranked
    together by their mass (both directions sum to last_q, so the masses are
    directly comparable).  For a threshold tau the kept set is band 0 plus
    every candidate with mass >= tau.  The oracle keeps the set of the
    largest candidate tau whose active entries reach ``density`` of the
    causal entries; if no tau does, every positive candidate is kept."""
    v = np.asarray(v, np.float64)
    S = np.asarray(S, np.float64)
    target = density * total_causal_entries(L)

    def sets(tau):
        Ss = np.concatenate([[0], 1 + np.flatnonzero(S[1:] >= tau)]).astype(np.int64)
        Vs = np.flatnonzero(v >= tau).astype(np.int64)
        return Vs, Ss

    def A(tau):
        Vs, Ss = sets(tau)
        return active_entries(L, Vs, Ss, bs)

    if A(np.inf) >= target:
        return sets(np.inf)
    cand = np.unique(np.concatenate([S[1:], v]))
    cand = cand[cand > 0][::-1]                       # descending
    lo, hi = 0, cand.size - 1                          # A(cand[i]) non-decreasing in i
    if A(cand[hi]) < target:
        return sets(cand[hi])
    while lo < hi:
        mid = (lo + hi) // 2
        if A(cand[mid]) >= target:
            hi = mid
        else:
            lo = mid + 1
    return sets(cand[lo])


def build_index(Q, K, last_q: int, top_p: float, scale: float | None = None,
                stripes: int = 1, block: int = 64, density: float = 0.0, index_mode: int = 0):
    """Per query head (V_h, S_h): ascending kept verticals (token ids) and
    kept slash bands (band 0 always included).  ``density > 0`` selects by
    budget fill instead of top-p; ``index_mode = 1`` then gives every head
    its GQA group's union (``group_shared_index``).  Returns (index list, v, S)."""
    L = Q.shape[0]
    bs = block * stripes
    v, S = index_scores(Q, K, last_q, scale, stripes, block)
    index = []
    for h in range(v.shape[0]):
        if density > 0:
            Vh, Sh = select_budget(v[h], S[h], L, bs, density)
        else:
            Vh = select_top_p(v[h], top_p)
            Sh = np.union1d(select_top_p(S[h], top_p), [0]).astype(np.int64)
        index.append((Vh, Sh))
    if index_mode == 1:
        index = group_shared_index(index, Q.shape[1] // K.shape[1])
    return index, v, S


def group_shared_index(index, G: int):
    """GQA-group-shared index ([MT] 三/核心创新/2, the kernel-aware granularity
    trade-off): every query head of a key/value group (heads g G .. g G + G - 1)
    gets the union of the group's kept verticals and the union of its kept
    bands (band 0 stays kept).  Returns a new per-head list."""
    out = []
    for g in range(len(index) // G):
        heads = index[g * G:(g + 1) * G]
        Vu = np.unique(np.concatenate([np.asarray(V, np.int64) for V, _ in heads]))
        Su = np.unique(np.concatenate([np.asarray(S, np.int64) for _, S in heads] + [np.array([0])]))
        out.extend([(Vu, Su)] * G)
    return out


# ----------------------------------------------------------------------------
# The VS mask and masked attention ([MT] 三/核心创新/2 "Ring Attention with the
# sparse index": only the active entries of the sub-matrix are computed)

def _row_mask(rows: np.ndarray, L: int, Vh, Sh, bs: int) -> np.ndarray:
    m = np.arange(L)
    nbs = L // bs
    inS = np.zeros(nbs, bool)
    inS[np.asarray(Sh, np.int64)] = True
    isV = np.zeros(L, bool)
    isV[np.asarray(Vh, np.int64)] = True
    band = (rows // bs)[:, None] - (m // bs)[None, :]
    causal = m[None, :] <= rows[:, None]
    return causal & (inS[np.clip(band, 0, nbs - 1)] | isV[None, :])


def explicit_mask(L: int, Vh, Sh, bs: int = 64) -> np.ndarray:
    """Dense boolean [L, L] mask of one head (small L only)."""
    return _row_mask(np.arange(L), L, Vh, Sh, bs)


def _chunks(L: int, rows: np.ndarray, budget: int = 1 << 23):
    step = max(1, budget // max(L, 1))
    for i in range(0, rows.size, step):
        yield rows[i:i + step]


def attention_forward_rows(Q, K, V, index, rows, scale=None, stripes=1, block=64):
    """Masked softmax attention for the listed query rows only.

    O_n = sum_{m active} softmax_m(scale q_n . k_m) v_m and
    LSE_n = log sum_{m active} exp(scale q_n . k_m), per head.
    Returns O [len(rows), Hq, d] and LSE [Hq, len(rows)]."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    rows = np.asarray(rows, np.int64)
    O = np.zeros((rows.size, Hq, d))
    LSE = np.zeros((Hq, rows.size))
    for h in range(Hq):
        Vh, Sh = index[h]
        kh, vh = K[:, h // G, :], V[:, h // G, :]
        off = 0
        for r in _chunks(L, rows):
            msk = _row_mask(r, L, Vh, Sh, bs)
            s = np.where(msk, scale * (Q[r, h, :] @ kh.T), -np.inf)
            mx = s.max(axis=1, keepdims=True)
            p = np.exp(s - mx)
            l = p.sum(axis=1, keepdims=True)
            O[off:off + r.size, h, :] = (p @ vh) / l
            LSE[h, off:off + r.size] = (mx + np.log(l))[:, 0]
            off += r.size
    return O, LSE


def attention_forward(Q, K, V, index, scale=None, stripes=1, block=64):
    """All rows of ``attention_forward_rows``: O [L, Hq, d], LSE [Hq, L]."""
    return attention_forward_rows(Q, K, V, index, np.arange(Q.shape[0]), scale, stripes, block)


def attention_backward(Q, K, V, dO, index, scale=None, stripes=1, block=64):
    """Gradients of the masked attention (mask held fixed) for cotangent dO.

    Per head with P the masked softmax: dV = P^T dO, dP = dO V^T,
    dS = P * (dP - rowsum(P * dP)), dQ = scale dS K, dK = scale dS^T Q;
    dK and dV of a key/value head sum over the query heads that share it."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        Vh, Sh = index[h]
        g = h // G
        kh, vh = K[:, g, :], V[:, g, :]
        for r in _chunks(L, np.arange(L)):
            msk = _row_mask(r, L, Vh, Sh, bs)
            s = np.where(msk, scale * (Q[r, h, :] @ kh.T), -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dP = dO[r, h, :] @ vh.T
            dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
            dV[:, g, :] += p.T @ dO[r, h, :]
            dQ[r, h, :] = scale * (dS @ kh)
            dK[:, g, :] += scale * (dS.T @ Q[r, h, :])
    return dQ, dK, dV


def attention_backward_dkdv_keys(Q, K, V, dO, index, keys, scale=None, stripes=1, block=64):
    """dK and dV of the listed key rows only (same definitions as
    ``attention_backward``): each query row n whose mask reaches one of the
    keys takes its full masked softmax P_n, dP_n = dO_n V^T and
    dS_n = P_n * (dP_n - P_n . dP_n), and adds P_nm dO_n to dV_m and
    scale dS_nm q_n to dK_m, summed over the query heads of the key's group.
    The rows visited are a superset of those reaching the keys (rows outside
    a key's mask add zero there): the row tiles ``t + B`` for each listed
    key's tile t and kept band B, and, when a listed key is a kept vertical,
    every row from that key on.  Returns dK, dV [len(keys), Hkv, d]."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    L, Hq, d = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    nbs = L // bs
    keys = np.asarray(keys, np.int64)
    dK = np.zeros((keys.size, Hkv, d))
    dV = np.zeros((keys.size, Hkv, d))
    for h in range(Hq):
        Vh, Sh = index[h]
        g = h // G
        kh, vh = K[:, g, :], V[:, g, :]
        tiles = (np.unique(keys // bs)[:, None] + np.asarray(Sh, np.int64)[None, :]).ravel()
        tiles = np.unique(tiles[tiles < nbs])
        rows = (tiles[:, None] * bs + np.arange(bs)[None, :]).ravel()
        vert = keys[np.isin(keys, np.asarray(Vh, np.int64))]
        if vert.size:
            rows = np.union1d(rows, np.arange(vert.min(), L))
        for r in _chunks(L, rows):
            msk = _row_mask(r, L, Vh, Sh, bs)
            s = np.where(msk, scale * (Q[r, h, :] @ kh.T), -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dP = dO[r, h, :] @ vh.T
            dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
            dV[:, g, :] += p[:, keys].T @ dO[r, h, :]
            dK[:, g, :] += scale * (dS[:, keys].T @ Q[r, h, :])
    return dK, dV


def attention_backward_bf16_products(Q, K, V, dO, index, scale=None, stripes=1, block=64):
    """``attention_backward`` with the roundings of an implementation whose
    tensor-core products take bf16 operands and accumulate in higher
    precision (the precision reading: bf16 inputs, fp32 accumulation,
    probabilities rounded to bf16 before they enter a product).  The
    definitions are unchanged; exactly three values are rounded to bf16,
    everything else is fp64:
      * O, the forward output, is stored as bf16 and D_n = sum_c dO_nc O_nc
        is formed from the stored O;
      * P enters dV = P^T dO as bf16;
      * dS = P * (dP - D) (with the unrounded P) enters dQ = scale dS K and
        dK = scale dS^T Q as bf16.
    It measures what that arithmetic itself costs, so a kernel that follows
    it can be held to a per-element tolerance."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        Vh, Sh = index[h]
        g = h // G
        kh, vh = K[:, g, :], V[:, g, :]
        for r in _chunks(L, np.arange(L)):
            msk = _row_mask(r, L, Vh, Sh, bs)
            s = np.where(msk, scale * (Q[r, h, :] @ kh.T), -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            O_b = bf16_round(p @ vh)
            D = (dO[r, h, :] * O_b).sum(axis=1, keepdims=True)
            dP = dO[r, h, :] @ vh.T
            dS_b = bf16_round(p * (dP - D))
            dV[:, g, :] += bf16_round(p).T @ dO[r, h, :]
            dQ[r, h, :] = scale * (dS_b @ kh)
            dK[:, g, :] += scale * (dS_b.T @ Q[r, h, :])
    return dQ, dK, dV


# ----------------------------------------------------------------------------
# Striped sparse ring attention ([MT] 三/核心创新/3 "平衡稀疏环注意力": striped
# layout over W workers; [RA] §2.1 block-wise ring computation with an
# incremental softmax, §3.1 striped round-robin layout)

def _ring_step_mask(Ls, W, r, s, Vh, Sh, block):
    """Active entries of ring step (worker r, KV shard s) in local
    coordinates: worker r holds global tokens n = i W + r, shard s holds
    m = j W + s.  Local causal rule: j <= i when s <= r, else j < i (the
    global rule m <= n).  The shared index: slash band floor(i / block) -
    floor(j / block) kept (tiles of the shard-local order), or m a kept
    vertical."""
    i = np.arange(Ls)[:, None]
    j = np.arange(Ls)[None, :]
    causal = (j <= i) if s <= r else (j < i)
    nb = Ls // block
    inS = np.zeros(nb, bool)
    inS[np.asarray(Sh, np.int64)] = True
    band = i // block - j // block
    isV = np.zeros(Ls, bool)
    Vh = np.asarray(Vh, np.int64)
    isV[(Vh[Vh % W == s] - s) // W] = True
    return causal & (inS[np.clip(band, 0, nb - 1)] | isV[None, :].repeat(Ls, 0))


def striped_ring_forward(Q, K, V, index, W, scale=None, block=64):
    """Sparse ring attention over W striped workers, step by step.

    Worker r holds the queries of tokens r, r + W, ...; at step t it holds
    KV shard s = (r - t) mod W and folds that step's active entries into its
    running (M, l, O) (max, sum of exponentials, unnormalised output):
    M' = max(M, max s), l' = l e^(M - M') + sum e^(s - M'),
    O' = O e^(M - M') + sum e^(s - M') v.  After W steps O / l is the output
    and M + ln l the log-sum-exp.  ``index`` is the shared striped index
    (slash bands in shard-local 64 x 64 tiles, verticals as global tokens).
    Returns O [L, Hq, d] and LSE [Hq, L] in the global token order."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    Ls = L // W
    O = np.zeros_like(Q)
    LSE = np.zeros((Hq, L))
    for h in range(Hq):
        Vh, Sh = index[h]
        g = h // G
        for r in range(W):
            q = Q[r::W, h, :]
            M = np.full(Ls, -np.inf)
            l = np.zeros(Ls)
            acc = np.zeros((Ls, d))
            for t in range(W):
                sh = (r - t) % W
                msk = _ring_step_mask(Ls, W, r, sh, Vh, Sh, block)
                sc = np.where(msk, scale * (q @ K[sh::W, g, :].T), -np.inf)
                mx = np.maximum(M, sc.max(axis=1))
                live = np.isfinite(mx)
                f = np.where(live, np.exp(np.where(live, M - mx, 0.0)), 0.0)
                p = np.where(msk, np.exp(sc - np.where(live, mx, 0.0)[:, None]), 0.0)
                l = l * f + p.sum(axis=1)
                acc = acc * f[:, None] + p @ V[sh::W, g, :]
                M = mx
            O[r::W, h, :] = acc / l[:, None]
            LSE[h, r::W] = M + np.log(l)
    return O, LSE


def striped_ring_backward(Q, K, V, dO, index, W, scale=None, block=64):
    """Gradients of ``striped_ring_forward``, step by step in the same ring
    order: with the final O and LSE of every query, D_n = sum_c dO_nc O_nc;
    at step (r, s) P = exp(scale q k - LSE) on the step's active entries,
    dV_s += P^T dO_r, dS = P (dO_r V_s^T - D), dQ_r += scale dS K_s,
    dK_s += scale dS^T Q_r (dK, dV summed over the query heads of a group)."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    Ls = L // W
    O, LSE = striped_ring_forward(Q, K, V, index, W, scale, block)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        Vh, Sh = index[h]
        g = h // G
        for r in range(W):
            q, do = Q[r::W, h, :], dO[r::W, h, :]
            D = (do * O[r::W, h, :]).sum(axis=1, keepdims=True)
            lse = LSE[h, r::W][:, None]
            for t in range(W):
                sh = (r - t) % W
                msk = _ring_step_mask(Ls, W, r, sh, Vh, Sh, block)
                k, v = K[sh::W, g, :], V[sh::W, g, :]
                p = np.where(msk, np.exp(scale * (q @ k.T) - lse), 0.0)
                dS = p * (do @ v.T - D)
                dV[sh::W, g, :] += p.T @ do
                dQ[r::W, h, :] += scale * (dS @ k)
                dK[sh::W, g, :] += scale * (dS.T @ q)
    return dQ, dK, dV


def attention_backward_dq_rows(Q, K, V, dO, index, rows, scale=None, stripes=1, block=64):
    """dQ of the listed query rows only (same definitions as
    ``attention_backward``): per row n, P_n = masked softmax,
    dP_n = dO_n V^T, dS_n = P_n * (dP_n - P_n . dP_n), dQ_n = scale dS_n K."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    dO = np.asarray(dO, np.float64)
    L, Hq, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bs = block * stripes
    rows = np.asarray(rows, np.int64)
    dQ = np.zeros((rows.size, Hq, d))
    for h in range(Hq):
        Vh, Sh = index[h]
        kh, vh = K[:, h // G, :], V[:, h // G, :]
        off = 0
        for r in _chunks(L, rows):
            msk = _row_mask(r, L, Vh, Sh, bs)
            s = np.where(msk, scale * (Q[r, h, :] @ kh.T), -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dP = dO[r, h, :] @ vh.T
            dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
            dQ[off:off + r.size, h, :] = scale * (dS @ kh)
            off += r.size
    return dQ
