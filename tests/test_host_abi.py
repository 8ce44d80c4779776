"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments before any
launch (no GPU needed: validation returns before touching CUDA)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def vs():
    from dynamic_sparse_attention_index_gb300 import build as b
    b.build()
    import dynamic_sparse_attention_index_gb300 as m
    m.lib()
    return m


def test_exports_match_header(vs):
    hdr = open(os.path.join(ROOT, "include", "vs.h")).read()
    declared = set(re.findall(r"^\s*VS_API\s+(?:vs_status|size_t|const char\*)\s+(vs_\w+)\s*\(", hdr, re.M))
    assert declared == set(vs.EXPORTED)
    for name in declared:
        assert hasattr(vs.lib(), name)


def test_status_strings(vs):
    for c in range(7):
        assert vs.vs_status_string(c).startswith("VS_")


def test_workspace_sizes(vs):
    p = vs.make_params(131072, 16, 2, 128)
    for op in (vs.VS_OP_INDEX, vs.VS_OP_FWD, vs.VS_OP_BWD):
        assert vs.vs_workspace_bytes(p, op) >= 256
    assert vs.vs_workspace_bytes(p, vs.VS_OP_ROPE) == 0
    bad = vs.make_params(131072, 16, 3, 128)
    assert vs.vs_workspace_bytes(bad, vs.VS_OP_INDEX) == 0


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on these paths


def _call_index(vs, p, q=FAKE, k=FAKE, ws=FAKE, ws_bytes=1 << 40, ix=None):
    if ix is None:
        ix = vs.vs_index(FAKE, FAKE, FAKE, FAKE, None, None, None)
    return vs.lib().vs_index_build(ctypes.byref(p), q, k, ctypes.byref(ix), ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hkv=3), "VS_ERR_INVALID_ARG"),
    (dict(d=96), "VS_ERR_UNSUPPORTED"),
    (dict(block=32), "VS_ERR_UNSUPPORTED"),
    (dict(last_q=0), "VS_ERR_INVALID_ARG"),
    (dict(last_q=4097), "VS_ERR_INVALID_ARG"),
    (dict(top_p=0.0), "VS_ERR_INVALID_ARG"),
    (dict(top_p=1.5), "VS_ERR_INVALID_ARG"),
    (dict(L=4000), "VS_ERR_INVALID_ARG"),
    (dict(stripes=3), "VS_ERR_INVALID_ARG"),
    (dict(density=-0.1), "VS_ERR_INVALID_ARG"),
    (dict(index_mode=2), "VS_ERR_INVALID_ARG"),
    (dict(rope_mode=2), "VS_ERR_INVALID_ARG"),
    (dict(rope_mode=1, rope_theta=1.0), "VS_ERR_INVALID_ARG"),          # the adjoint needs the frequencies
    (dict(rope_mode=1, yarn_factor=32.0, yarn_orig_len=0), "VS_ERR_INVALID_ARG"),
])
def test_index_rejects_bad_params(vs, kw, code):
    args = dict(L=4096, Hq=4, Hkv=2, d=64, last_q=64, top_p=0.9)
    args.update(kw)
    p = vs.make_params(**args)
    assert _call_index(vs, p) == getattr(vs, code)


def test_index_rejects_bad_pointers_and_workspace(vs):
    p = vs.make_params(4096, 4, 2, 64)
    assert _call_index(vs, p, q=None) == vs.VS_ERR_INVALID_ARG
    assert _call_index(vs, p, q=FAKE + 2) == vs.VS_ERR_INVALID_ARG       # misaligned
    assert _call_index(vs, p, ix=vs.vs_index(None, FAKE, FAKE, FAKE, None, None, None)) == vs.VS_ERR_INVALID_ARG
    assert _call_index(vs, p, ix=vs.vs_index(FAKE, FAKE, FAKE, FAKE, FAKE + 4, None, None)) == vs.VS_ERR_INVALID_ARG
    assert _call_index(vs, p, ws=None) == vs.VS_ERR_WORKSPACE
    assert _call_index(vs, p, ws=FAKE + 16) == vs.VS_ERR_WORKSPACE       # not 256-aligned
    assert _call_index(vs, p, ws_bytes=16) == vs.VS_ERR_WORKSPACE


def test_attention_rejects_bad_args(vs):
    L = vs.lib()
    p = vs.make_params(4096, 4, 2, 64)
    ix = vs.vs_index(FAKE, FAKE, FAKE, FAKE, None, None, None)
    r = L.vs_sparse_attn_fwd(ctypes.byref(p), ctypes.byref(ix), FAKE, FAKE, None, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == vs.VS_ERR_INVALID_ARG
    r = L.vs_sparse_attn_fwd(ctypes.byref(p), ctypes.byref(ix), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, None)
    assert r == vs.VS_ERR_WORKSPACE
    p128 = vs.make_params(4096, 4, 2, 128)
    r = L.vs_sparse_attn_bwd(ctypes.byref(p128), ctypes.byref(ix), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, None, FAKE, 1 << 40, None)
    assert r == vs.VS_ERR_INVALID_ARG
    d64 = vs.make_params(4096, 4, 2, 64)
    assert vs.vs_workspace_bytes(d64, vs.VS_OP_BWD) == 0
    r = L.vs_sparse_attn_bwd(ctypes.byref(d64), ctypes.byref(ix), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == vs.VS_ERR_UNSUPPORTED  # the backward is built for d = 128 only; rejected before any launch
    bad = vs.make_params(4096, 4, 2, 80)
    r = L.vs_sparse_attn_fwd(ctypes.byref(bad), ctypes.byref(ix), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == vs.VS_ERR_UNSUPPORTED


def test_rope_rejects_bad_args(vs):
    L = vs.lib()
    p = vs.make_params(4096, 4, 2, 64, rope_theta=1.0)
    assert L.vs_rope(ctypes.byref(p), 4, FAKE, FAKE, 0, None) == vs.VS_ERR_INVALID_ARG
    p = vs.make_params(4096, 4, 2, 64, yarn_factor=32.0, yarn_orig_len=0)
    assert L.vs_rope(ctypes.byref(p), 4, FAKE, FAKE, 0, None) == vs.VS_ERR_INVALID_ARG


def test_bwd_workspace_sizes():
    """The backward's minimum workspace, and the room it suggests for
    stored dS tiles (64 x 64 bf16 blocks, per head 1.5 x the density's share
    of the causal blocks plus four vertical chunks per query block; none for
    top-p selection; every head in one pass up to 32 GiB, else the fewest
    passes over key/value head groups up to 96 GiB a pass, else none; and
    one block of zeros)."""
    import dynamic_sparse_attention_index_gb300 as vs
    L, Hq = 131072, 16
    nb = L // 64
    p0 = vs.make_params(L, Hq, 2, 128)
    mn = vs.vs_workspace_bytes(p0, vs.VS_OP_BWD_MIN)
    assert mn > 0 and vs.vs_workspace_bytes(p0, vs.VS_OP_BWD) == mn
    p5 = vs.make_params(L, Hq, 2, 128, density=0.05)
    assert vs.vs_workspace_bytes(p5, vs.VS_OP_BWD_MIN) == mn
    extra = vs.vs_workspace_bytes(p5, vs.VS_OP_BWD) - mn
    cap = int(1.5 * 0.05 * nb * (nb + 1) / 2 + 4 * nb) + 1
    tables = Hq * (nb + 2 * nb) * 4  # band ranks (one per band, W = 1) and two block bases per query block
    zero = 8192  # one block of zeros after the heads' blocks
    assert Hq * cap * 8192 + zero + tables <= extra <= Hq * cap * 8192 + zero + tables + 4 * 256
    big = vs.make_params(1 << 20, 32, 8, 128, density=0.05)
    assert vs.vs_workspace_bytes(big, vs.VS_OP_BWD) == vs.vs_workspace_bytes(big, vs.VS_OP_BWD_MIN)
    # 512K, 32 / 8 heads: 20.9 GB of blocks a head; one group of four heads a pass
    L5, Hq5 = 1 << 19, 32
    nb5 = L5 // 64
    p5 = vs.make_params(L5, Hq5, 8, 128, density=0.05)
    mn5 = vs.vs_workspace_bytes(p5, vs.VS_OP_BWD_MIN)
    extra = vs.vs_workspace_bytes(p5, vs.VS_OP_BWD) - mn5
    cap = int(1.5 * 0.05 * nb5 * (nb5 + 1) / 2 + 4 * nb5) + 1
    tables = Hq5 * (nb5 + 2 * nb5) * 4
    assert 4 * cap * 8192 + zero + tables <= extra <= 4 * cap * 8192 + zero + tables + 4 * 256
    # 128K, 16 / 8 heads at density 0.1: 42.3 GB for all heads (over 32 GiB), two
    # passes of four groups
    p6 = vs.make_params(L, Hq, 8, 128, density=0.1)
    extra = vs.vs_workspace_bytes(p6, vs.VS_OP_BWD) - vs.vs_workspace_bytes(p6, vs.VS_OP_BWD_MIN)
    cap = int(1.5 * 0.1 * nb * (nb + 1) / 2 + 4 * nb) + 1
    assert Hq * cap * 8192 > 32 * 2 ** 30
    tables = Hq * (nb + 2 * nb) * 4
    assert 8 * cap * 8192 + zero + tables <= extra <= 8 * cap * 8192 + zero + tables + 4 * 256


def _call_xattn(vs, p, stride=8, thr=0.9, q=FAKE, k=FAKE, ws=FAKE, ws_bytes=1 << 40, out=None):
    if out is None:
        out = vs.vs_xattn_index(FAKE, FAKE, None, None)
    return vs.lib().vs_xattn_index_build(ctypes.byref(p), stride, thr, q, k, ctypes.byref(out), ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(stride=3), "VS_ERR_INVALID_ARG"),        # not a power of two
    (dict(stride=0), "VS_ERR_INVALID_ARG"),
    (dict(stride=128), "VS_ERR_INVALID_ARG"),      # does not divide bs = 64
    (dict(stride=32), "VS_ERR_UNSUPPORTED"),       # two strided rows per block
    (dict(thr=0.0), "VS_ERR_INVALID_ARG"),
    (dict(thr=1.5), "VS_ERR_INVALID_ARG"),
    (dict(q=None), "VS_ERR_INVALID_ARG"),
    (dict(k=FAKE + 8), "VS_ERR_INVALID_ARG"),
    (dict(ws=None), "VS_ERR_WORKSPACE"),
    (dict(ws_bytes=1024), "VS_ERR_WORKSPACE"),
])
def test_xattn_rejects_bad_args(vs, kw, code):
    p = vs.make_params(4096, 4, 2, 128)
    assert _call_xattn(vs, p, **kw) == getattr(vs, code)


def test_xattn_rejects_missing_outputs_and_sizes_workspace(vs):
    p = vs.make_params(4096, 4, 2, 128)
    assert _call_xattn(vs, p, out=vs.vs_xattn_index(None, FAKE, None, None)) == vs.VS_ERR_INVALID_ARG
    assert _call_xattn(vs, p, out=vs.vs_xattn_index(FAKE, None, None, None)) == vs.VS_ERR_INVALID_ARG
    assert _call_xattn(vs, p, out=vs.vs_xattn_index(FAKE, FAKE, FAKE + 4, None)) == vs.VS_ERR_INVALID_ARG
    # stride 1 (full-resolution cells, 64 rows per block) is accepted up to the argument checks
    n = vs.vs_workspace_bytes(p, vs.VS_OP_XATTN)
    assert n >= 4 * 4096 * 8  # a (max, sum) per strided row at stride 1
    assert _call_xattn(vs, p, stride=1, ws_bytes=n - 256) == vs.VS_ERR_WORKSPACE
    # striped tiles: bs = 64 W, the stride must keep 4 .. 128 strided rows per block
    p32 = vs.make_params(65536, 2, 1, 128, stripes=32)
    assert _call_xattn(vs, p32, stride=8) == vs.VS_ERR_UNSUPPORTED  # 256 rows per block
    assert vs.vs_workspace_bytes(vs.make_params(4096, 4, 3, 128), vs.VS_OP_XATTN) == 0
