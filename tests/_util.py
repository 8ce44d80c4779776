"""Test helpers: tensor conversion and index-set comparison (no method arithmetic)."""
import numpy as np

import synth


def to_dev(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def f64(bits):
    return synth.bf16_bits_to_f64(bits)


def bf16_bits_of(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_index_lists(ix, Hq):
    out = []
    vc, sc = ix.v_cnt.cpu().numpy(), ix.s_cnt.cpu().numpy()
    vi, si = ix.v_idx.cpu().numpy(), ix.s_idx.cpu().numpy()
    for h in range(Hq):
        out.append((vi[h, :vc[h]].astype(np.int64), si[h, :sc[h]].astype(np.int64)))
    return out


def topp_sets_agree(x_or, sel_or, sel_gpu, p, tol=1e-6, forced=()):
    """True if the GPU selection equals the oracle's, except for elements at
    the top-p threshold: each element in the symmetric difference must have a
    normalised mass within `tol` of the oracle's threshold element, or sit at
    a cumulative normalised mass within `tol` of p."""
    a, b = set(sel_or.tolist()), set(sel_gpu.tolist())
    diff = (a ^ b) - set(forced)
    if not diff:
        return True, []
    tot = x_or.sum()
    xn = x_or / tot
    kept = np.array(sorted(a - set(forced)), dtype=np.int64)
    thr = xn[kept].min() if kept.size else 0.0
    order = np.argsort(-x_or, kind="stable")
    cum = np.cumsum(xn[order])
    rank = np.empty_like(order)
    rank[order] = np.arange(order.size)
    bad = []
    for e in diff:
        near_thr = abs(xn[e] - thr) <= tol
        c_before = cum[rank[e]] - xn[e]
        near_p = abs(c_before - p) <= tol or abs(cum[rank[e]] - p) <= tol
        if not (near_thr or near_p):
            bad.append((e, xn[e], thr))
    return not bad, bad


def inject_index(vs, p, index, dev):
    """Device IndexBuffers holding a given per-head (V_h, S_h) index."""
    import torch
    ix = vs.IndexBuffers.allocate(p, dev, scores=False)
    nbs = p.L // (p.block * p.stripes)
    vi = np.zeros((p.Hq, p.L), np.int32)
    si = np.zeros((p.Hq, nbs), np.int32)
    vc = np.zeros(p.Hq, np.int32)
    sc = np.zeros(p.Hq, np.int32)
    for h, (Vh, Sh) in enumerate(index):
        vi[h, :len(Vh)] = Vh
        si[h, :len(Sh)] = Sh
        vc[h], sc[h] = len(Vh), len(Sh)
    ix.v_idx.copy_(torch.from_numpy(vi))
    ix.s_idx.copy_(torch.from_numpy(si))
    ix.v_cnt.copy_(torch.from_numpy(vc))
    ix.s_cnt.copy_(torch.from_numpy(sc))
    return ix


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def budget_sets_agree(v_or, S_or, kept_or, kept_gpu, tol=1e-6):
    """True if a budget-fill selection on the GPU equals the oracle's fp64
    one except for candidates at the threshold: every vertical or band
    (band 0 is forced on both sides) in the symmetric difference must have
    a normalised mass (mass / total mass of its direction) within `tol` of
    the oracle's threshold, the smallest kept candidate mass, normalised the
    same way."""
    (Vo, So), (Vg, Sg) = kept_or, kept_gpu
    tv, ts = v_or.sum(), S_or.sum()
    masses = [v_or[Vo] / tv] + ([S_or[So[So > 0]] / ts] if (So > 0).any() else [])
    thr = min(float(m.min()) for m in masses if m.size) if any(m.size for m in masses) else 0.0
    bad = []
    for e in set(Vo.tolist()) ^ set(Vg.tolist()):
        if abs(v_or[e] / tv - thr) > tol:
            bad.append(("v", e, v_or[e] / tv, thr))
    for e in (set(So.tolist()) ^ set(Sg.tolist())) - {0}:
        if abs(S_or[e] / ts - thr) > tol:
            bad.append(("s", e, S_or[e] / ts, thr))
    return not bad, bad


def ulp_bf16(x):
    """Spacing of bf16 values at |x| (2^(e - 7) for |x| in [2^e, 2^(e+1)))."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 2.0 ** -133)


def grad_close(name, got, ref, emu):
    """Backward parity, element by element.  ``ref`` is the exact fp64
    gradient, ``emu`` the same gradient with the bf16 roundings of the
    stated arithmetic (oracle.attention_backward_bf16_products).  The kernel
    must follow that arithmetic: every element within 2e-2 + half a bf16 ulp
    of ``emu`` (the output is stored as bf16); and the result must be close
    to the exact gradient: relative L2 <= 1e-2, every element within
    2e-2 + half an ulp of ``ref`` plus the arithmetic's own distance
    |emu - ref| at that element."""
    err_e = np.abs(got - emu)
    bad = err_e > 2e-2 + 0.5 * ulp_bf16(emu)
    assert not bad.any(), (name, "vs bf16-products oracle", int(bad.sum()), float(err_e.max()))
    err = np.abs(got - ref)
    bad = err > 2e-2 + 0.5 * ulp_bf16(ref) + np.abs(emu - ref)
    assert not bad.any(), (name, "vs exact oracle", int(bad.sum()), float(err.max()))
    assert rel_l2(got, ref) <= 1e-2, (name, rel_l2(got, ref))
