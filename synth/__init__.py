"""Seeded synthetic inputs for the vertical-slash (VS) sparse attention workloads.

This module is shared by the oracle-side tests and the CUDA-side tests and
bench.  It holds random-number generation and the workload recipes only:
none of the attention method's arithmetic (no RoPE, no softmax, no index
selection) lives here.

Generator: a counter-based SplitMix64 stream.  Element ``i`` of stream
``seed`` is ``mix64(mix64(seed) + (i + 1) * 0x9E3779B97F4A7C15)`` where
``mix64`` is the SplitMix64 finaliser (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  Normals come
from the Box-Muller transform on pairs of consecutive uniforms, in fp64,
then are rounded fp64 -> fp32 -> bf16, each step round-to-nearest-even.

Why no RoPE here: every configuration asks for "RoPE'd N(0,1)" queries and
keys.  A RoPE rotation is orthogonal, so a rotated vector of i.i.d. N(0,1)
entries is again i.i.d. N(0,1); such tensors are drawn directly.  Outlier
scaling multiplies a whole key row and commutes with the rotation.  The one
recipe whose structure depends on RoPE (a per-head constant bias added
*before* rotation) is returned un-rotated, and each side applies its own RoPE.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids inside one workload: seed = 1000 * workload_id + tensor_id
T_Q, T_K, T_V, T_DO, T_OUTLIER, T_BIAS = 0, 1, 2, 3, 4, 5


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed: int) -> np.uint64:
    return _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def uniform_bits(seed: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs ``start .. start+count-1`` of stream ``seed``."""
    key = _stream_key(seed)
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + ctr * _GOLDEN)


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniforms in (0, 1]: (top 53 bits + 1) * 2^-53, fp64."""
    b = uniform_bits(seed, start, count) >> np.uint64(11)
    return (b.astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _normal_chunk(seed: int, pair0: int, npairs: int) -> np.ndarray:
    u = uniform01(seed, 2 * pair0, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out


def normal_f64(seed: int, n: int, threads: int | None = None) -> np.ndarray:
    """``n`` standard normals of stream ``seed`` (fp64), element order fixed."""
    npairs = (n + 1) // 2
    chunk = 1 << 20
    starts = list(range(0, npairs, chunk))
    out = np.empty(2 * npairs, dtype=np.float64)

    def work(p0):
        m = min(chunk, npairs - p0)
        out[2 * p0: 2 * (p0 + m)] = _normal_chunk(seed, p0, m)

    nt = threads or min(len(starts), os.cpu_count() or 1)
    if nt <= 1 or len(starts) == 1:
        for p0 in starts:
            work(p0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, starts))
    return out[:n]


def normal_bf16_rows(seed: int, shape, transform=None, rows_per_chunk: int | None = None) -> np.ndarray:
    """bf16 bit patterns of ``normal_f64(seed, prod(shape))`` reshaped to
    ``shape``, built a block of rows at a time so that the fp64 copy of a
    large tensor never exists whole.  ``transform(block, r0)`` may change a
    block of rows (starting at row ``r0``) in fp64 before rounding.  The
    result is bit-identical to rounding the whole fp64 tensor at once (both
    steps are elementwise and the stream is addressed by element index)."""
    shape = tuple(shape)
    row = int(np.prod(shape[1:]))
    if rows_per_chunk is None:
        rows_per_chunk = max(2, (1 << 24) // max(row, 1))
    rows_per_chunk += rows_per_chunk % 2          # even element offsets keep Box-Muller pairs whole
    out = np.empty(shape, dtype=np.uint16)
    starts = list(range(0, shape[0], rows_per_chunk))

    def work(r0):
        r1 = min(shape[0], r0 + rows_per_chunk)
        e0, e1 = r0 * row, r1 * row
        p0 = e0 // 2
        blk = _normal_chunk(seed, p0, (e1 - 2 * p0 + 1) // 2)[e0 - 2 * p0: e1 - 2 * p0]
        blk = blk.reshape((r1 - r0,) + shape[1:])
        if transform is not None:
            blk = transform(blk, r0)
        out[r0:r1] = f64_to_bf16_bits(blk)

    nt = min(len(starts), os.cpu_count() or 1)
    if nt <= 1:
        for r0 in starts:
            work(r0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, starts))
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def permutation_prefix(seed: int, n: int, k: int) -> np.ndarray:
    """First ``k`` entries of a seeded random permutation of range(n) (sorted)."""
    keys = uniform_bits(seed, 0, n)
    order = np.argsort(keys, kind="stable")
    return np.sort(order[:k]).astype(np.int64)


@dataclass
class Workload:
    """One synthetic problem.  Tensors are bf16 bit patterns, token-major
    ``[L, H, d]`` (batch 1).  ``q_rope``/``k_rope`` say whether a RoPE
    rotation with ``rope_theta`` (and YaRN settings) still has to be applied
    by the consumer: False means the tensors already follow the rotated
    distribution."""
    name: str
    L: int
    Hq: int
    Hkv: int
    d: int
    last_q: int
    top_p: float
    backward: bool
    rope_theta: float
    yarn_factor: float
    yarn_orig_len: int
    needs_rope: bool
    stripes: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray | None
    outliers: np.ndarray
    meta: dict = field(default_factory=dict)


# The five workload recipes (id -> spec).  Shapes, value distributions and
# index parameters follow the configurations the headline numbers are quoted
# on; everything is synthetic.
RECIPES = {
    1: dict(name="mha1_L4096_d64_fwd", L=4096, Hq=1, Hkv=1, d=64, last_q=64, top_p=0.9,
            backward=False, theta=1e4, outlier_count=8, outlier_scale=8.0, bias=False,
            yarn=1.0, stripes=1),
    2: dict(name="mha8_L32768_d128_fwd_localbias", L=32768, Hq=8, Hkv=8, d=128, last_q=64,
            top_p=0.95, backward=False, theta=1e4, outlier_frac=0.001, outlier_scale=6.0,
            bias=True, yarn=1.0, stripes=1),
    3: dict(name="gqa16x2_L131072_d128_fwdbwd", L=131072, Hq=16, Hkv=2, d=128, last_q=64,
            top_p=0.95, backward=True, theta=1e4, outlier_frac=0.001, outlier_scale=6.0,
            bias=False, yarn=1.0, stripes=1),
    4: dict(name="gqa16x2_L262144_d128_fwdbwd_striped32", L=262144, Hq=16, Hkv=2, d=128,
            last_q=64, top_p=0.95, backward=True, theta=1e4, outlier_frac=0.001,
            outlier_scale=6.0, bias=False, yarn=1.0, stripes=32),
    5: dict(name="gqa32x8_L524288_d128_fwdbwd_yarn32", L=524288, Hq=32, Hkv=8, d=128,
            last_q=64, top_p=0.95, backward=True, theta=5e5, outlier_frac=0.0005,
            outlier_scale=8.0, bias=False, yarn=32.0, stripes=1),
}


def make_workload(wid: int, L: int | None = None, Hq: int | None = None,
                  Hkv: int | None = None, d: int | None = None,
                  last_q: int | None = None, top_p: float | None = None,
                  stripes: int | None = None, backward: bool | None = None,
                  seed_base: int | None = None) -> Workload:
    """Build workload ``wid`` (1..5), optionally shrunk (same distributions).

    Seeds: ``1000 * seed_base + tensor_id`` with ``seed_base`` defaulting to
    the workload id.
    """
    r = dict(RECIPES[wid])
    L = L or r["L"]
    Hq = Hq or r["Hq"]
    Hkv = Hkv or r["Hkv"]
    d = d or r["d"]
    last_q = last_q or r["last_q"]
    top_p = r["top_p"] if top_p is None else top_p
    stripes = stripes or r["stripes"]
    backward = r["backward"] if backward is None else backward
    sb = wid if seed_base is None else seed_base
    s = lambda t: 1000 * sb + t

    if "outlier_count" in r:
        n_out = r["outlier_count"]
    else:
        n_out = max(1, int(round(r["outlier_frac"] * L)))
    outl = permutation_prefix(s(T_OUTLIER), L, min(n_out, L))
    meta = {}
    bq = bk = None
    if r["bias"]:
        # per-head constant added to every channel of q and k before RoPE;
        # beta_h ~ U[0.25, 0.5]
        bq = 0.25 + 0.25 * uniform01(s(T_BIAS), 0, Hq)
        G = Hq // Hkv
        bk = bq.reshape(Hkv, G).mean(axis=1)
        meta["beta_q"] = bq
        meta["beta_k"] = bk
    is_out = np.zeros(L, bool)
    is_out[outl] = True

    def q_tf(blk, r0):
        if bq is not None:
            blk += bq[None, :, None]
        return blk

    def k_tf(blk, r0):
        if bk is not None:
            blk += bk[None, :, None]
        # outlier keys: whole row (all KV heads) scaled
        rows = is_out[r0:r0 + blk.shape[0]]
        blk[rows] *= r["outlier_scale"]
        return blk

    q = normal_bf16_rows(s(T_Q), (L, Hq, d), q_tf)
    k = normal_bf16_rows(s(T_K), (L, Hkv, d), k_tf)
    v = normal_bf16_rows(s(T_V), (L, Hkv, d))
    do = normal_bf16_rows(s(T_DO), (L, Hq, d)) if backward else None
    return Workload(
        name=r["name"], L=L, Hq=Hq, Hkv=Hkv, d=d, last_q=last_q, top_p=top_p,
        backward=backward, rope_theta=r["theta"], yarn_factor=r["yarn"],
        yarn_orig_len=int(L // r["yarn"]) if r["yarn"] > 1 else 0,
        needs_rope=bool(r["bias"]), stripes=stripes,
        q=q, k=k, v=v, do=do, outliers=outl, meta=meta)


def normal_bf16(seed: int, shape) -> np.ndarray:
    """Convenience: bf16 bit patterns of i.i.d. N(0,1), given shape."""
    n = int(np.prod(shape))
    return f64_to_bf16_bits(normal_f64(seed, n)).reshape(shape)
