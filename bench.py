"""Benchmark: one training step of the vertical-slash sparse attention hot path.

Workload (default): the 128K GQA training shape, 16 query / 2 key-value heads,
d = 128, L = 131072, batch 1, bf16, synthetic seeded inputs (N(0,1) queries,
keys and values with 0.1 % outlier keys at 6x norm, dO ~ N(0,1)).

One step = every stage of the path on one batch:
  RoPE(Q), RoPE(K) -> sparse index (last 64 queries, budget fill to the
  pages' 95 % sparsity operating point) -> sparse attention forward ->
  backward (D, dK/dV, dQ) -> RoPE adjoint on dQ, dK.
Metric: effective TFLOP/s of sparse attention fwd+bwd = 14 d A / step time,
A = exact active (query, key) entries (fwd 4 d A + bwd 10 d A), with the
index and RoPE time inside the step.

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
For N > 1 (torchrun, one rank per GPU) every rank runs an independent
replica of the step (the path has no cross-GPU exchange): value sums the
ranks' FLOPs over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

WORKLOADS = {
    # name -> (recipe id, overrides); forward-only recipes time RoPE, index and forward
    "gqa16x2_L131072_d128_fwdbwd": (3, {}),
    "gqa16x2_L32768_d128_fwdbwd": (3, {"L": 32768}),   # small case for profiling
    # striped layout emulation: 32 round-robin shards (slash tiles of 64 x 32 tokens)
    "gqa16x2_L262144_d128_striped32_fwdbwd": (4, {}),
    "gqa16x2_L65536_d128_striped32_fwdbwd": (4, {"L": 65536}),
    # single head, L = 4096, d = 64, forward only (8 outlier keys x 8)
    "mha1_L4096_d64_fwd": (1, {}),
    # 8-head MHA, L = 32768, forward only, per-head slash-shaped local bias
    "mha8_L32768_d128_fwd_localbias": (2, {}),
    # Llama-3.1-8B attention shape: GQA 32/8, L = 524288, YaRN x32 (base 5e5)
    "gqa32x8_L524288_d128_fwdbwd_yarn32": (5, {}),
}
DENSITY = 0.05     # budget fill: 95 % sparsity (fixed in the pages' experiments)
LAST_Q, TOP_P = 64, 0.95
# library kernels per step: RoPE of Q and K; the index (two tensor-core
# scoring passes, slash sums, selection); the forward (three prep kernels,
# attention); the backward (three prep kernels, D, dK / dV for the vertical
# and the slash units, the recomputing dQ kernel, and with rope_mode = 1 the
# RoPE adjoint on dK and the one on dQ, which returns at once when the dQ
# kernel of the stored dS tiles applied it in its epilogue)
KERNELS_PER_STEP = {"rope": 2, "index": 4, "fwd": 4, "bwd": 9}
KERNELS_PER_STEP_FWD = {"rope": 2, "index": 4, "fwd": 4}
# ex2.approx issue rate of one SM per clock (the index's exponentials;
# measured with a standalone microbenchmark on this GPU)
MUFU_EX2_PER_CLK_SM = 32
N_SM = 152
# DRAM bytes of one backward call (dram__bytes_read.sum + dram__bytes_write.sum
# over its kernels, from a one-pass ncu capture of the workload), read from the
# profile summary together with the SHA-256 of the kernel sources it was taken
# on: when the sources have changed since, the figure no longer applies and
# the line reports null.
TRAFFIC_SOURCES = ("attn_bwd.cu", "attn_fwd.cu", "attn_prep.cu", "attn_dq_stored.cu", "attn_common.cuh", "ptx.cuh",
                   "common.cuh")


def kernel_sources_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "dynamic_sparse_attention_index_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def bwd_traffic_bytes(workload: str):
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}_backward.txt")
    try:
        kv = dict(ln.split(None, 1) for ln in open(path) if ln.strip() and not ln.startswith("#"))
    except (OSError, ValueError):
        return None
    if kv.get("kernel_sources_sha256", "").strip() != kernel_sources_sha():
        return None
    return int(kv["bytes_per_backward_call"])


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return {"bf16_tflops": m["bf16_tflops"], "bf16_tflops_sustained": m["bf16_tflops_sustained"],
                "hbm_gbs": m["hbm_gbs"], "src": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist(backend: str = "nccl"):
    """Process group of a torchrun launch (one rank per GPU), or none."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        dist.init_process_group(backend)
        return dist, rank, local, ws
    return None, 0, 0, 1


def replica_throughput(dist, world, flops_per_rank, ms, e2e_ms, device):
    """Whole-job throughput of independent replicas: every rank did the same
    work, the job takes as long as the slowest rank (max over ranks), and
    the value is world x work / that time (TFLOP/s).  Returns (value, e2e
    value, ms, e2e ms) with the times taken over all ranks."""
    import torch
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms, e2e_ms = t.tolist()
    return (world * flops_per_rank / (ms * 1e-3) / 1e12, world * flops_per_rank / (e2e_ms * 1e-3) / 1e12, ms,
            e2e_ms)


def index_roofline(w, A_index_time_ms, kept, pk, sm_mhz):
    """Index build against its binding roof.  Algorithmic work of one build
    (the minimum the method needs): K read once, the last_q query rows read,
    the vertical and slash masses written once and read once by the
    selection, the kept lists written; one QK^T over the last_q rows
    (2 d last_q Hq L flop) and one exponential per score (last_q Hq L).
    The roof is the largest of the three times at the measured HBM and bf16
    peaks and the ex2 rate (MUFU_EX2_PER_CLK_SM x SMs x the maximum SM
    clock)."""
    L, Hq, Hkv, d, q = w.L, w.Hq, w.Hkv, w.d, LAST_Q
    nbs = L // (64 * w.stripes)
    bytes_ = 2 * L * Hkv * d + 2 * q * Hq * d + 2 * 4 * Hq * (L + nbs) + 4 * kept
    flops = 2.0 * d * q * Hq * L
    exps = float(q * Hq * L)
    mufu = MUFU_EX2_PER_CLK_SM * N_SM * sm_mhz * 1e6          # ex2 per second
    t = {"hbm": bytes_ / (pk["hbm_gbs"] * 1e9), "tensor": flops / (pk["bf16_tflops"] * 1e12),
         "alu": exps / mufu}
    bound = max(t, key=t.get)
    sec = A_index_time_ms * 1e-3
    ach = {"hbm": bytes_ / sec / 1e9, "tensor": flops / sec / 1e12, "alu": exps / sec / 1e12}[bound]
    peak = {"hbm": pk["hbm_gbs"], "tensor": pk["bf16_tflops"], "alu": mufu / 1e12}[bound]
    unit = {"hbm": "GB/s", "tensor": "TFLOP/s", "alu": "Tex2/s"}[bound]
    return {"kernel": "vs_index_build (scores, row statistics, slash bands, selection)", "bound": bound,
            "achieved": round(ach, 3), "peak": round(peak, 3), "unit": unit, "frac": round(ach / peak, 4),
            "algorithmic": {"bytes": int(bytes_), "flop": flops, "ex2": exps},
            "roof_us": {k: round(v * 1e6, 2) for k, v in t.items()}, "index_us": round(A_index_time_ms * 1e3, 2),
            "peak_src": pk["src"] + (" HBM copy" if bound == "hbm" else " bf16 burst" if bound == "tensor"
                                     else " ex2 rate x SMs x max SM clock")}


def xattn_ablation(vs, torch, w, Q, K, dev, stream, pk, stride: int, threshold: float, iters: int = 5):
    """The anti-diagonal block index (the pages' "w/ XAttn Idx." ablation) on
    the same RoPE'd Q and K, timed alone after the step's timed region: ms per
    call, and its tensor work against the bf16 burst peak.  Counted work: the
    causal strided cells of both passes, 2 x 2 S d FLOP each per head."""
    W = w.stripes
    bs = 64 * W
    S = stride if bs // stride <= 128 else bs // 128
    px = vs.make_params(w.L, w.Hq, w.Hkv, w.d, stripes=W)
    xi = vs.XattnBuffers.allocate(px, dev)
    ws = vs.workspace(px, vs.VS_OP_XATTN, dev)
    for _ in range(3):
        vs.vs_xattn_index_build(px, S, threshold, Q, K, xi, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        vs.vs_xattn_index_build(px, S, threshold, Q, K, xi, ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    R = w.L // S
    flop = 2.0 * (R * (R + 1) // 2) * 2 * S * w.d * w.Hq
    tf = flop / (ms * 1e-3) / 1e12
    act = int(xi.active_entries.sum().item())
    st = vs.vs_device_status(ws)
    del xi, ws
    return {"kernel": "vs_xattn_index_build (two tcgen05 scoring passes, block selection)", "stride": S,
            "block": bs, "threshold": threshold, "ms": round(ms, 4), "achieved": round(tf, 2), "unit": "TFLOP/s",
            "bound": "tensor", "peak": pk["bf16_tflops"], "frac": round(tf / pk["bf16_tflops"], 4),
            "peak_src": pk["src"] + " bf16 burst", "flop": flop,
            "sparsity": round(1 - act / (w.Hq * w.L * (w.L + 1) / 2), 5),
            "device_status": vs.vs_status_string(st), "launches_per_call": 3}


def run_gpu(args):
    import torch

    import dynamic_sparse_attention_index_gb300 as vs
    from dynamic_sparse_attention_index_gb300 import build as vsbuild

    dist, rank, local, world = _dist()
    vsbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wid, ov = WORKLOADS[args.workload]
    w = synth.make_workload(wid, **ov)
    L, Hq, Hkv, d = w.L, w.Hq, w.Hkv, w.d
    W = w.stripes
    bwd = w.backward
    rope_kw = dict(rope_theta=w.rope_theta, yarn_factor=w.yarn_factor, yarn_orig_len=w.yarn_orig_len)
    imode = 1 if args.index_mode == "group" else 0
    # the backward returns the gradients of the un-rotated Q and K (rope_mode = 1)
    p = vs.make_params(L, Hq, Hkv, d, last_q=LAST_Q, top_p=TOP_P, density=DENSITY, stripes=W, index_mode=imode,
                       rope_mode=1 if bwd else 0, **rope_kw)
    p_nat = vs.make_params(L, Hq, Hkv, d, last_q=LAST_Q, top_p=TOP_P, density=0.0, stripes=W, index_mode=imode,
                           **rope_kw)

    def pinned(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    h_in = [pinned(w.q), pinned(w.k), pinned(w.v)] + ([pinned(w.do)] if bwd else [])
    d_in = [t.to(dev) for t in h_in]
    Qr, Kr, V = d_in[:3]
    Q, K = torch.empty_like(Qr), torch.empty_like(Kr)
    O = torch.empty_like(Q)
    lse = torch.empty((Hq, L), dtype=torch.float32, device=dev)
    d_out = [torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)] if bwd else [O]
    ix = vs.IndexBuffers.allocate(p, dev)
    ws_i = vs.workspace(p, vs.VS_OP_INDEX, dev)
    ring = W > 1  # striped layout: the W-worker ring, run step by step
    ws_f = vs.workspace(p, vs.VS_OP_RING_FWD if ring else vs.VS_OP_FWD, dev)
    ws_b = vs.workspace(p, vs.VS_OP_RING_BWD if ring else vs.VS_OP_BWD, dev) if bwd else None
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out]
    stream = torch.cuda.current_stream()
    phases = ("rope", "index", "fwd", "bwd") if bwd else ("rope", "index", "fwd")
    ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in phases}

    step_ev = {}  # ring: per-step events of one instrumented pass ("fwd", "bwd" -> W * W + 1 events)

    def step(timed=False, io=None, before_bwd=None):
        # io: the step's input and output device buffers; before_bwd: called
        # right before the backward (the end-to-end loop waits there for dO)
        ins, outs = io if io is not None else (d_in, d_out)
        qr, kr, v_ = ins[:3]

        def rec(k, i):
            if timed:
                ev[k][i].record(stream)
        rec("rope", 0)
        vs.vs_rope(p, Hq, qr, Q, False)
        vs.vs_rope(p, Hkv, kr, K, False)
        rec("rope", 1)
        rec("index", 0)
        vs.vs_index_build(p, Q, K, ix, ws_i)
        rec("index", 1)
        rec("fwd", 0)
        if ring:
            vs.vs_striped_ring_fwd(p, ix, Q, K, v_, O if bwd else outs[0], lse, ws_f, events=step_ev.get("fwd"))
        else:
            vs.vs_sparse_attn_fwd(p, ix, Q, K, v_, O if bwd else outs[0], lse, ws_f)
        rec("fwd", 1)
        if bwd:
            dq, dk, dv = outs
            if before_bwd is not None:
                before_bwd()
            rec("bwd", 0)
            if ring:
                vs.vs_striped_ring_bwd(p, ix, Q, K, v_, O, lse, ins[3], dq, dk, dv, ws_b, events=step_ev.get("bwd"))
            else:
                vs.vs_sparse_attn_bwd(p, ix, Q, K, v_, O, lse, ins[3], dq, dk, dv, ws_b)
            rec("bwd", 1)

    # natural top-p sparsity (reported; not the timed operating point)
    vs.vs_rope(p, Hq, Qr, Q, False)
    vs.vs_rope(p, Hkv, Kr, K, False)
    ix_nat = vs.IndexBuffers.allocate(p_nat, dev)
    vs.vs_index_build(p_nat, Q, K, ix_nat, vs.workspace(p_nat, vs.VS_OP_INDEX, dev))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    T = L * (L + 1) // 2
    A = int(ix.active_entries.sum().item())
    A_nat = int(ix_nat.active_entries.sum().item())
    kept = int(ix.v_cnt.sum().item() + ix.s_cnt.sum().item())
    del ix_nat
    balance = None
    if W > 1:
        # per-shard work of the striped layout against contiguous and ZigZag
        # splits of the contiguous (W = 1) index built on the same inputs
        p1 = vs.make_params(L, Hq, Hkv, d, last_q=LAST_Q, top_p=TOP_P, density=DENSITY, **rope_kw)
        ix1 = vs.IndexBuffers.allocate(p1, dev)
        vs.vs_index_build(p1, Q, K, ix1, vs.workspace(p1, vs.VS_OP_INDEX, dev))
        ix_w = vs.IndexBuffers.allocate(p, dev)
        vs.vs_index_build(p, Q, K, ix_w, vs.workspace(p, vs.VS_OP_INDEX, dev))
        torch.cuda.synchronize()
        balance = shard_balance(L, W, index_lists(ix_w, Hq), index_lists(ix1, Hq))
        balance["timed"] = ring_balance(vs, p1, ix1, Q, K, V, W, dev, step, step_ev, bwd)
        del ix1, ix_w
    # the backward's status word says how dQ was formed (1: from the dS
    # tiles stored in its workspace, 0: S and dP recomputed) and in how many
    # passes over key/value head groups
    dq_stored = bool(ws_b is not None and not ring and int(ws_b[8:12].view(torch.int32).item()) == 1)
    dq_passes = int(ws_b[12:16].view(torch.int32).item()) if dq_stored else 0
    assert vs.vs_device_status(ws_f) == vs.VS_OK
    assert ws_b is None or vs.vs_device_status(ws_b) == vs.VS_OK

    sampler = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    # per-phase averages over K extra steps (events on every step)
    acc = {k: 0.0 for k in ev}
    for _ in range(args.steps):
        step(timed=True)
        torch.cuda.synchronize()
        for k in ev:
            acc[k] += ev[k][0].elapsed_time(ev[k][1])
    phase = {k: v / args.steps for k, v in acc.items()}
    clocks = sampler.stop()
    # every bounded in-kernel wait of the timed steps completed (a wait that
    # gave up would leave VS_ERR_TIMEOUT and its site in a status word)
    dev_status = {k: vs.vs_status_string(vs.vs_device_status(ws))
                  for k, ws in (("index", ws_i), ("fwd", ws_f), ("bwd", ws_b)) if ws is not None}

    # End to end through the C ABI with host buffers: every step copies its
    # inputs (Q, K, V and, with a backward, dO) in from pinned host memory and
    # its results (dQ, dK, dV, or O for a forward-only step) back out.  The
    # copies run on their own streams over two sets of device and host
    # buffers, so one step's transfers overlap its neighbours' kernels, as a
    # training loop's input pipeline would; the timed region runs from the
    # first copy in to the last copy out.
    io = [(d_in, d_out), ([torch.empty_like(t) for t in d_in], [torch.empty_like(t) for t in d_out])]
    hout = [h_out, [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in h_out]]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # Q, K and V (what RoPE, the index and the forward read) are copied in
    # first; dO, read only by the backward, arrives under the forward
    in_done = [torch.cuda.Event() for _ in range(2)]
    do_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def e2e_steps(n):
        s_in.wait_event(e0)
        for i in range(n):
            b = i & 1
            ins, outs = io[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])  # step i - 2 no longer reads these inputs
                for dst, src in zip(ins[:3], h_in[:3]):
                    dst.copy_(src, non_blocking=True)
                in_done[b].record(s_in)
                for dst, src in zip(ins[3:], h_in[3:]):
                    dst.copy_(src, non_blocking=True)
                do_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if i >= 2:
                stream.wait_event(out_done[b])  # step i - 2's results were copied out
            step(io=(ins, outs), before_bwd=lambda b=b: stream.wait_event(do_done[b]))
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for dst, src in zip(hout[b], outs):
                    dst.copy_(src, non_blocking=True)
                out_done[b].record(s_out)
        for b in range(min(2, n)):
            stream.wait_event(out_done[b])

    # one untimed pass over both buffer sets first (first use of the copy
    # streams and of the second set of pinned host buffers)
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_steps(min(2, args.steps))
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    flops = (14.0 if bwd else 4.0) * d * A
    value, e2e_val, ms, e2e_ms = replica_throughput(dist, world, flops, ms, e2e_ms, dev)
    pk = _peaks()
    xattn = None
    if args.xattn_stride > 0:
        # after the timed regions: Q and K hold the last step's rotated inputs
        xattn = xattn_ablation(vs, torch, w, Q, K, dev, stream, pk, args.xattn_stride, args.xattn_threshold)
    fwd_tf = 4.0 * d * A / (phase["fwd"] * 1e-3) / 1e12
    bwd_tf = 10.0 * d * A / (phase["bwd"] * 1e-3) / 1e12 if bwd else None
    # dominant call: the backward (dK/dV + dQ kernels, 10 d A) when there is
    # one, else the forward (4 d A); each phase lasts milliseconds, so the
    # burst peak is the denominator (the sustained one is listed beside it)
    dom = ("vs_sparse_attn_bwd (dK/dV + dQ)", bwd_tf) if bwd else ("vs_sparse_attn_fwd", fwd_tf)
    peak, peak_s = pk["bf16_tflops"], pk["bf16_tflops_sustained"]
    kps = dict(KERNELS_PER_STEP if bwd else KERNELS_PER_STEP_FWD)
    if dq_stored:
        # the dS plan and, per pass over KV-head groups, the dQ kernel that
        # reads the tiles (the recomputing one returns at once) and, after
        # the first pass, the two dK / dV kernels again
        kps["bwd"] += 1 + dq_passes + 2 * (dq_passes - 1)
    if ring:
        # ring setup (shard lists, band bitmaps, a vertical union and packed
        # rows per shard) and W x W steps: one forward kernel per step; D, the
        # two dK / dV kernels and the dQ kernel per step, two final casts, the
        # RoPE adjoint on dQ and dK
        kps["fwd"] = 2 + 2 * W + W * W
        if bwd:
            kps["bwd"] = 1 + 2 + 2 * W + 3 * W * W + 2 + 2
    out = {
        "metric": "VS sparse attn fwd+bwd ms and effective TFLOP/s at 128K (% bf16 peak)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "L": L, "Hq": Hq, "Hkv": Hkv, "d": d, "batch": 1,
                   "pass": "fwd+bwd" if bwd else "fwd", "last_q": LAST_Q,
                   "index": f"budget fill to density {DENSITY}"
                            + (", shared by each GQA group (union of its heads' sets)" if imode else ""),
                   "sparsity": round(1 - A / (Hq * T), 5),
                   "natural_top_p_sparsity": round(1 - A_nat / (Hq * T), 5), "top_p": TOP_P,
                   "active_entries": A, "l2": "inputs larger than L2 (no flush)" if L * Hq * d * 2 > 2 * (126 << 20)
                   else "no flush (inputs smaller than L2)", "stripes": W,
                   "rope": {"theta": w.rope_theta, "yarn_factor": w.yarn_factor},
                   "parallelism": f"replicas x{world}"},
        "breakdown_ms": {k: round(v, 4) for k, v in phase.items()},
        **({"shard_balance": balance} if balance else {}),
        "fwd_tflops": round(fwd_tf, 2), **({"bwd_tflops": round(bwd_tf, 2)} if bwd else {}),
        "index_overhead": round(phase["index"] / max(ms, 1e-9), 4),
        "roofline": {"kernel": dom[0], "bound": "tensor",
                     "achieved": round(dom[1], 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(dom[1] / peak, 4), "traffic": bwd_traffic_bytes(args.workload) if bwd else None,
                     "peak_src": pk["src"] + " bf16 burst",
                     "frac_of_sustained": round(dom[1] / peak_s, 4)},
        "index_roofline": index_roofline(w, phase["index"], kept, pk, clocks.get("sm_max_mhz") or 2070.0),
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "copies": "own streams, two buffer sets, dO under the forward",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": sum(kps.values()) * args.steps,
        "clocks": clocks,
        "device_status": dev_status,
        **({"dq_path": (f"stored dS tiles ({dq_passes} passes)" if dq_passes > 1 else "stored dS tiles")
                        if dq_stored else "recomputed S and dP"} if bwd and not ring else {}),
        **({"xattn_index": xattn} if xattn else {}),
    }
    if rank == 0 and not args.no_cpu_baseline:
        rows = max(16, int(args.cpu_rows * (131072 / L) * (16 / Hq)))
        out["cpu_baseline"] = cpu_baseline(w, index_lists(ix, Hq), d, min(rows, args.cpu_rows), bwd)
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def index_lists(ix, Hq):
    vc, sc = ix.v_cnt.cpu().numpy(), ix.s_cnt.cpu().numpy()
    vi, si = ix.v_idx.cpu().numpy(), ix.s_idx.cpu().numpy()
    return [(vi[h, :vc[h]].astype(np.int64), si[h, :sc[h]].astype(np.int64)) for h in range(Hq)]


def row_active_counts(L, V, S, bs):
    """Active causal entries of every query row of one head under a VS index:
    kept slash bands S (band n//bs - m//bs, band 0 always kept) plus kept
    verticals V outside kept bands (the mask the kernels compute)."""
    nbs = L // bs
    kept = np.zeros(nbs, bool)
    kept[np.asarray(S, np.int64)] = True
    kept[0] = True
    n = np.arange(L, dtype=np.int64)
    qb = n // bs
    kc = np.cumsum(kept) - 1                      # kept bands 1..b
    slash = kc[qb] * bs + (n - qb * bs + 1)
    cnt_v = np.bincount(np.asarray(V, np.int64) // bs, minlength=nbs)
    before = np.concatenate([[0], np.cumsum(cnt_v)[:-1]])   # verticals in earlier blocks
    inband = np.zeros(nbs, np.int64)                        # ... of those, in kept bands
    for B in np.flatnonzero(kept[1:]) + 1:
        inband[B:] += cnt_v[:nbs - B]
    return slash + (before - inband)[qb]


def ring_balance(vs, p1, ix1, Q, K, V, W, dev, step, step_ev, bwd):
    """Timed per-worker and per-step balance.  Striped layout: one step of
    the bench run with CUDA events around each of the W x W ring steps
    (worker r, step t); a worker's time is the sum of its W steps, a ring
    step's time the slowest worker's (the ring advances together).
    Contiguous and ZigZag splits of the contiguous index: each worker's rows
    of the forward, timed as one vs_sparse_attn_fwd_rows call (contiguous:
    rows [r L/W, (r+1) L/W); ZigZag: 2 W chunks, worker k holds chunks k and
    2 W - 1 - k)."""
    import torch
    from dynamic_sparse_attention_index_gb300 import ring_model as rm
    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(W * W + 1)]
    step_ev["fwd"] = mk()
    if bwd:
        step_ev["bwd"] = mk()
    step()
    torch.cuda.synchronize()
    out = {"unit": "ms (CUDA events)"}
    for k, ev in list(step_ev.items()):
        t = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(W * W)]).reshape(W, W)
        worker = t.sum(1)
        per_step = t.max(0)
        out[f"striped_ring_{k}"] = {
            "total_ms": round(float(t.sum()), 3), "worker_max_over_mean": round(float(worker.max() / worker.mean()), 4),
            "step_max_over_mean": round(float((t.max(0) / t.mean(0)).max()), 4),
            "step_ms_slowest_worker": [round(float(x), 4) for x in per_step]}
        if k == "fwd" and W == rm.PAGES_A100_4x8.workers:
            # the pages' hierarchical-ring model with these measured step times
            # and the pages' link times (4 nodes x 8 GPUs, NVLink 0.13 ms,
            # InfiniBand 0.98 ms per step)
            r = rm.forward_latency_ms([float(x) for x in per_step], rm.PAGES_A100_4x8)
            out["ring_model_fwd"] = {"topology": "4 nodes x 8, t_intra 0.13 ms, t_inter 0.98 ms",
                                     "flat_ms": round(r["flat_ms"], 3),
                                     "hierarchical_ms": round(r["hierarchical_ms"], 3),
                                     "flat_comm_bound_steps": r["flat"]["comm_bound_steps"],
                                     "hierarchical_exposed_outer_ms": round(r["hierarchical"]["exposed_outer_ms"], 3)}
    step_ev.clear()
    L = p1.L
    O = torch.empty_like(Q)
    lse = torch.empty((p1.Hq, L), dtype=torch.float32, device=dev)
    ws = vs.workspace(p1, vs.VS_OP_FWD, dev)
    Ls, Lz = L // W, L // (2 * W)

    def timed(ranges):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for lo, hi in ranges:
            vs.vs_sparse_attn_fwd_rows(p1, ix1, Q, K, V, O, lse, ws, lo, hi)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    timed([(0, Ls)])  # warm-up
    for name, workers in (("contiguous", [[(r * Ls, (r + 1) * Ls)] for r in range(W)]),
                          ("zigzag", [[(k * Lz, (k + 1) * Lz), ((2 * W - 1 - k) * Lz, (2 * W - k) * Lz)]
                                      for k in range(W)])):
        t = np.array([timed(rg) for rg in workers])
        out[f"{name}_fwd_rows"] = {"worker_max_over_mean": round(float(t.max() / t.mean()), 4),
                                   "worker_ms_max": round(float(t.max()), 4), "worker_ms_mean": round(float(t.mean()), 4)}
    return out


def shard_balance(L, W, index_striped, index_contig):
    """Work (active entries) per worker for W workers: the striped layout
    (worker r holds tokens r, r + W, ...; index with 64 W-token slash tiles)
    and the contiguous and ZigZag splits (2 W chunks, worker k holds chunks k
    and 2 W - 1 - k) of the contiguous index.  Returns max / mean of each."""
    striped = sum(row_active_counts(L, V, S, 64 * W) for V, S in index_striped).reshape(L // W, W).sum(0)
    rows = sum(row_active_counts(L, V, S, 64) for V, S in index_contig)
    contig = rows.reshape(W, L // W).sum(1)
    chunks = rows.reshape(2 * W, L // (2 * W)).sum(1)
    zigzag = chunks[:W] + chunks[::-1][:W]
    r = lambda a: round(float(a.max() / a.mean()), 4)
    return {"workers": W, "unit": "active entries per worker", "striped_max_over_mean": r(striped),
            "contiguous_max_over_mean": r(contig), "zigzag_max_over_mean": r(zigzag),
            "striped_total": int(striped.sum()), "contiguous_index_total": int(rows.sum())}


def cpu_baseline(w, index, d, nrows, bwd=True):
    """The fp64 oracle, as it stands, on a bounded sample of the step: the
    forward (and, for a training step, dQ) of `nrows` query rows spread over
    the sequence, every head.  Reported in TFLOP/s counting the work those
    calls do on the sampled rows' active entries: 4 d for the forward and
    6 d for dQ (S and dP recomputed, dS K); the rows' dK / dV contributions
    are not run."""
    import oracle
    f = synth.bf16_bits_to_f64
    rows = np.linspace(0, w.L - 1, nrows).astype(np.int64)

    def sampled(bits):
        # the oracle reads only the sampled query rows: the rest stay zero
        # pages that are never touched
        x = np.zeros(bits.shape, np.float64)
        x[rows] = f(bits[rows])
        return x
    Q, K, V = sampled(w.q), f(w.k), f(w.v)
    bs = 64 * w.stripes
    act = 0
    for (Vh, Sh) in index:
        inS = np.zeros(w.L // bs, bool)
        inS[Sh] = True
        isV = np.zeros(w.L, bool)
        isV[Vh] = True
        for n in rows:
            m = np.arange(n + 1)
            act += int((inS[n // bs - m // bs] | isV[m]).sum())
    t0 = time.perf_counter()
    oracle.attention_forward_rows(Q, K, V, index, rows, stripes=w.stripes)
    if bwd:
        oracle.attention_backward_dq_rows(Q, K, V, sampled(w.do), index, rows, stripes=w.stripes)
    dt = time.perf_counter() - t0
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count()
    per = 10 if bwd else 4
    what = "forward + dQ" if bwd else "forward"
    return {"value": round(per * d * act / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 {what} of {nrows} query rows x {w.Hq} heads ({act} active entries, "
                      f"{per} d flop each), {dt:.1f} s"}


def run_reference(args):
    """Reference arm: the fp64 CPU oracle timed on this machine's host cores."""
    dist, rank, local, world = (None, 0, 0, 1)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    wid, ov = WORKLOADS[args.workload]
    w = synth.make_workload(wid, **ov)
    f = synth.bf16_bits_to_f64
    Q, K = f(w.q), f(w.k)
    index, _, _ = oracle.build_index(Q, K, LAST_Q, TOP_P, density=DENSITY, stripes=w.stripes)
    vals = []
    base = None
    rows = max(4, int(args.cpu_rows // 8 * (131072 / w.L) * (16 / w.Hq)))
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, index, w.d, min(rows, args.cpu_rows), w.backward)
        if i >= args.warmup:
            vals.append(r["value"])
            base = r
    v = float(np.mean(vals))
    out = {"metric": "VS sparse attn fwd+bwd ms and effective TFLOP/s at 128K (% bf16 peak)",
           "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
           "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": args.workload, "index": f"budget fill to density {DENSITY}"},
           "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": base["cores"], "kind": "oracle",
                            "sample": base["sample"]},
           "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="gqa16x2_L131072_d128_fwdbwd", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--index-mode", default="head", choices=["head", "group"],
                    help="one index per query head (the method) or one per GQA group (union)")
    ap.add_argument("--xattn-stride", type=int, default=8,
                    help="stride of the anti-diagonal block index timed after the step (0: skip)")
    ap.add_argument("--xattn-threshold", type=float, default=0.9)
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
