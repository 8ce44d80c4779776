"""Python binding of the GB300 VS sparse attention library (libvs.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/vs.h``.  PyTorch supplies
device memory and the current stream.  There is no fallback: if the shared
library is missing or fails to load, every call raises.

Entry points mirror the C names: ``vs_workspace_bytes``, ``vs_rope``,
``vs_index_build``, ``vs_index_build_noalloc``, ``vs_sparse_attn_fwd``, ``vs_sparse_attn_bwd``,
``vs_sparse_attn_fwd_rows``, ``vs_striped_ring_fwd``, ``vs_striped_ring_bwd``, ``vs_device_status``,
``vs_status_string``, ``vs_xattn_index_build``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvs.so")

VS_OK, VS_ERR_INVALID_ARG, VS_ERR_UNSUPPORTED, VS_ERR_WORKSPACE, VS_ERR_CUDA, VS_ERR_TIMEOUT, VS_ERR_BOUNDS = range(7)
VS_OP_INDEX, VS_OP_FWD, VS_OP_BWD, VS_OP_ROPE, VS_OP_RING_FWD, VS_OP_RING_BWD, VS_OP_BWD_MIN, VS_OP_XATTN = range(8)

#: every symbol the header declares
EXPORTED = ("vs_workspace_bytes", "vs_status_string", "vs_rope", "vs_index_build",
            "vs_index_build_noalloc", "vs_sparse_attn_fwd", "vs_sparse_attn_bwd", "vs_device_status",
            "vs_striped_ring_fwd", "vs_striped_ring_bwd", "vs_sparse_attn_fwd_rows", "vs_xattn_index_build")

#: size of the static scratch behind vs_index_build_noalloc (VS_INDEX_NOALLOC_SCRATCH_BYTES)
INDEX_NOALLOC_SCRATCH_BYTES = 8 << 20


class VSError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {vs_status_string(code)}")


class vs_params(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("last_q", ctypes.c_int32), ("top_p", ctypes.c_float), ("block", ctypes.c_int32),
        ("stripes", ctypes.c_int32), ("softmax_scale", ctypes.c_float), ("density", ctypes.c_float),
        ("rope_theta", ctypes.c_double), ("yarn_factor", ctypes.c_float), ("yarn_orig_len", ctypes.c_int32),
        ("index_mode", ctypes.c_int32), ("rope_mode", ctypes.c_int32),
    ]


class vs_index(ctypes.Structure):
    _fields_ = [
        ("v_idx", ctypes.c_void_p), ("v_cnt", ctypes.c_void_p), ("s_idx", ctypes.c_void_p),
        ("s_cnt", ctypes.c_void_p), ("v_score", ctypes.c_void_p), ("s_score", ctypes.c_void_p),
        ("active_entries", ctypes.c_void_p),
    ]


class vs_xattn_index(ctypes.Structure):
    _fields_ = [
        ("block_score", ctypes.c_void_p), ("block_mask", ctypes.c_void_p), ("block_cnt", ctypes.c_void_p),
        ("active_entries", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libvs.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run dynamic_sparse_attention_index_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, VP, SZ = ctypes.POINTER(vs_params), ctypes.POINTER(vs_index), ctypes.c_void_p, ctypes.c_size_t
        i32 = ctypes.c_int32
        L.vs_workspace_bytes.argtypes = [P, ctypes.c_int]
        L.vs_workspace_bytes.restype = SZ
        L.vs_status_string.argtypes = [ctypes.c_int]
        L.vs_status_string.restype = ctypes.c_char_p
        L.vs_rope.argtypes = [P, i32, VP, VP, i32, VP]
        L.vs_index_build.argtypes = [P, VP, VP, I, VP, SZ, VP]
        L.vs_index_build_noalloc.argtypes = [P, VP, VP, I, VP]
        L.vs_sparse_attn_fwd.argtypes = [P, I, VP, VP, VP, VP, VP, VP, SZ, VP]
        L.vs_sparse_attn_bwd.argtypes = [P, I, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]
        L.vs_device_status.argtypes = [VP, VP]
        EV = ctypes.POINTER(ctypes.c_void_p)
        L.vs_striped_ring_fwd.argtypes = [P, I, VP, VP, VP, VP, VP, VP, SZ, EV, i32, VP]
        L.vs_sparse_attn_fwd_rows.argtypes = [P, I, VP, VP, VP, VP, VP, VP, SZ, i32, i32, VP]
        L.vs_striped_ring_bwd.argtypes = [P, I, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, EV, i32, VP]
        L.vs_xattn_index_build.argtypes = [P, i32, ctypes.c_float, VP, VP, ctypes.POINTER(vs_xattn_index), VP,
                                           SZ, VP]
        for f in ("vs_rope", "vs_index_build", "vs_index_build_noalloc", "vs_sparse_attn_fwd",
                  "vs_sparse_attn_bwd", "vs_device_status", "vs_striped_ring_fwd", "vs_striped_ring_bwd",
                  "vs_sparse_attn_fwd_rows", "vs_xattn_index_build"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


#: index_mode values
VS_INDEX_PER_HEAD, VS_INDEX_GROUP_SHARED = 0, 1


def make_params(L, Hq, Hkv, d, last_q=64, top_p=0.95, stripes=1, softmax_scale=0.0, density=0.0,
                rope_theta=10000.0, yarn_factor=1.0, yarn_orig_len=0, block=64, index_mode=0,
                rope_mode=0) -> vs_params:
    return vs_params(L, Hq, Hkv, d, last_q, top_p, block, stripes, softmax_scale, density,
                     rope_theta, yarn_factor, yarn_orig_len, index_mode, rope_mode)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != VS_OK:
        raise VSError(code, where)


def vs_status_string(code: int) -> str:
    return lib().vs_status_string(code).decode()


def vs_workspace_bytes(p: vs_params, op: int) -> int:
    return int(lib().vs_workspace_bytes(ctypes.byref(p), op))


@dataclass
class IndexBuffers:
    """Device arrays of one sparse index (see ``vs_index`` in include/vs.h)."""
    v_idx: object
    v_cnt: object
    s_idx: object
    s_cnt: object
    v_score: object = None
    s_score: object = None
    active_entries: object = None

    @classmethod
    def allocate(cls, p: vs_params, device, scores: bool = True):
        import torch
        nbs = p.L // (p.block * p.stripes)
        i32 = dict(dtype=torch.int32, device=device)
        return cls(
            v_idx=torch.empty((p.Hq, p.L), **i32), v_cnt=torch.zeros(p.Hq, **i32),
            s_idx=torch.empty((p.Hq, nbs), **i32), s_cnt=torch.zeros(p.Hq, **i32),
            v_score=torch.empty((p.Hq, p.L), dtype=torch.float32, device=device) if scores else None,
            s_score=torch.empty((p.Hq, nbs), dtype=torch.float32, device=device) if scores else None,
            active_entries=torch.zeros(p.Hq, dtype=torch.int64, device=device))

    def c(self) -> vs_index:
        return vs_index(*[(t.data_ptr() if t is not None else None) for t in
                          (self.v_idx, self.v_cnt, self.s_idx, self.s_cnt, self.v_score, self.s_score,
                           self.active_entries)])


@dataclass
class XattnBuffers:
    """Device arrays of one anti-diagonal block index (``vs_xattn_index``)."""
    block_score: object
    block_mask: object
    block_cnt: object = None
    active_entries: object = None

    @classmethod
    def allocate(cls, p: vs_params, device):
        import torch
        nb = p.L // (p.block * p.stripes)
        nw = (nb + 31) // 32
        return cls(block_score=torch.empty((p.Hq, nb, nb), dtype=torch.float32, device=device),
                   block_mask=torch.empty((p.Hq, nb, nw), dtype=torch.int32, device=device),
                   block_cnt=torch.empty((p.Hq, nb), dtype=torch.int32, device=device),
                   active_entries=torch.zeros(p.Hq, dtype=torch.int64, device=device))

    def c(self) -> vs_xattn_index:
        return vs_xattn_index(*[(t.data_ptr() if t is not None else None) for t in
                                (self.block_score, self.block_mask, self.block_cnt, self.active_entries)])

    def kept_blocks(self):
        """Host lists: per head, per block row I, the ascending kept block
        columns (decoded from the mask words)."""
        import numpy as np
        m = self.block_mask.cpu().numpy().view(np.uint32)
        Hq, nb, nw = m.shape
        bits = ((m[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(Hq, nb, nw * 32)[..., :nb]
        return [[np.flatnonzero(bits[h, I]).astype(np.int64) for I in range(nb)] for h in range(Hq)]


def workspace(p: vs_params, op: int, device):
    """A caller-owned scratch buffer for ``op`` (torch allocation)."""
    import torch
    n = max(vs_workspace_bytes(p, op), 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


def vs_rope(p: vs_params, H: int, x, y, transpose: bool = False, stream=None):
    _check(lib().vs_rope(ctypes.byref(p), H, _ptr(x), _ptr(y), int(transpose), _stream(stream)), "vs_rope")


def vs_index_build(p: vs_params, Q, K, index: IndexBuffers, ws, stream=None):
    ix = index.c()
    _check(lib().vs_index_build(ctypes.byref(p), _ptr(Q), _ptr(K), ctypes.byref(ix), _ptr(ws),
                                ws.numel(), _stream(stream)), "vs_index_build")


def vs_index_build_noalloc(p: vs_params, Q, K, index: IndexBuffers, stream=None):
    """vs_index_build on the library's static scratch: for callers that cannot
    hand over a workspace (see ``vs_index_build_noalloc`` in include/vs.h)."""
    ix = index.c()
    _check(lib().vs_index_build_noalloc(ctypes.byref(p), _ptr(Q), _ptr(K), ctypes.byref(ix), _stream(stream)),
           "vs_index_build_noalloc")


def vs_sparse_attn_fwd(p: vs_params, index: IndexBuffers, Q, K, V, O, lse, ws, stream=None):
    ix = index.c()
    _check(lib().vs_sparse_attn_fwd(ctypes.byref(p), ctypes.byref(ix), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                    _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), "vs_sparse_attn_fwd")


def vs_sparse_attn_fwd_rows(p: vs_params, index: IndexBuffers, Q, K, V, O, lse, ws, row_lo: int, row_hi: int,
                            stream=None):
    ix = index.c()
    _check(lib().vs_sparse_attn_fwd_rows(ctypes.byref(p), ctypes.byref(ix), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                         _ptr(lse), _ptr(ws), ws.numel(), row_lo, row_hi, _stream(stream)),
           "vs_sparse_attn_fwd_rows")


def vs_sparse_attn_bwd(p: vs_params, index: IndexBuffers, Q, K, V, O, lse, dO, dQ, dK, dV, ws, stream=None):
    ix = index.c()
    _check(lib().vs_sparse_attn_bwd(ctypes.byref(p), ctypes.byref(ix), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                    _ptr(lse), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(),
                                    _stream(stream)), "vs_sparse_attn_bwd")


def _events(events):
    if not events:
        return None, 0
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr, len(events)


def vs_striped_ring_fwd(p: vs_params, index: IndexBuffers, Q, K, V, O, lse, ws, events=None, stream=None):
    """Striped sparse ring forward (W = p.stripes workers, step by step);
    ``events``: optional list of W*W+1 torch.cuda.Event(enable_timing=True)
    recorded before every step and after the last."""
    ix = index.c()
    ev, n = _events(events)
    _check(lib().vs_striped_ring_fwd(ctypes.byref(p), ctypes.byref(ix), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                     _ptr(lse), _ptr(ws), ws.numel(), ev, n, _stream(stream)), "vs_striped_ring_fwd")


def vs_striped_ring_bwd(p: vs_params, index: IndexBuffers, Q, K, V, O, lse, dO, dQ, dK, dV, ws, events=None,
                        stream=None):
    ix = index.c()
    ev, n = _events(events)
    _check(lib().vs_striped_ring_bwd(ctypes.byref(p), ctypes.byref(ix), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                     _ptr(lse), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), ev,
                                     n, _stream(stream)), "vs_striped_ring_bwd")


def vs_device_status(ws, stream=None) -> int:
    return int(lib().vs_device_status(_ptr(ws), _stream(stream)))


def vs_xattn_index_build(p: vs_params, stride: int, threshold: float, Q, K, index: XattnBuffers, ws, stream=None):
    ix = index.c()
    _check(lib().vs_xattn_index_build(ctypes.byref(p), int(stride), float(threshold), _ptr(Q), _ptr(K),
                                      ctypes.byref(ix), _ptr(ws), ws.numel(), _stream(stream)),
           "vs_xattn_index_build")
