"""Step-time model of flat and hierarchical sparse ring attention.

MTraining review, section 三/核心创新/4 "分层稀疏环注意力" (hierarchical sparse
ring attention) and the forward-latency breakdown of its experiments
(计算-通信重叠分析): the context-parallel ring over W = nodes x gpus_per_node
workers moves one KV block per step while every worker computes on the block
it holds.

* Flat ring: the ring is synchronous and some hops cross nodes, so each of
  the first W - 1 steps lasts max(T_comp(t), T_inter); the last step only
  computes.  (The page: max{T_comp, T_intra, T_inter} = T_inter = 0.98 ms,
  31 steps, then 0.51 ms of final attention.)
* Hierarchical ring: an inner ring over the GPUs of a node (NVLink) walks
  the node's gpus_per_node KV blocks while an outer ring (InfiniBand) moves
  the next node's blocks in the background.  Inner step t lasts
  max(T_comp(t), T_intra); a round of gpus_per_node inner steps that has an
  outer transfer pending lasts at least T_inter.  (The page:
  max{T_comp, T_inner} = T_comp = 0.51 ms for all 32 steps.)

T_comp(t) is the compute time of ring step t, the slowest worker of that
step (the ring advances together).  On one GPU the striped ring runs the
W x W (worker, step) pairs one after another and times each
(``vs_striped_ring_fwd`` with step events); this module turns those
measured compute times into the multi-node step schedule the pages
describe.  It models communication only through the two link times; it
moves no data.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence


@dataclass(frozen=True)
class RingTopology:
    nodes: int
    gpus_per_node: int
    t_intra_ms: float   # one KV-block transfer between GPUs of a node
    t_inter_ms: float   # one KV-block transfer between nodes

    @property
    def workers(self) -> int:
        return self.nodes * self.gpus_per_node


#: The pages' measured setting: 4 nodes x 8 A100-40GB, NVLink 0.13 ms and
#: InfiniBand 0.98 ms per ring step.
PAGES_A100_4x8 = RingTopology(nodes=4, gpus_per_node=8, t_intra_ms=0.13, t_inter_ms=0.98)


def step_compute_ms(times_ms) -> list:
    """Per-step compute time of a synchronous ring from per-(worker, step)
    times ``times_ms[r][t]``: the slowest worker of each step."""
    W = len(times_ms)
    return [max(times_ms[r][t] for r in range(W)) for t in range(len(times_ms[0]))]


def flat_ring_ms(step_comp_ms: Sequence[float], topo: RingTopology) -> dict:
    """Flat ring: W - 1 communicating steps bounded by the slowest link,
    then one compute-only step."""
    W = len(step_comp_ms)
    link = topo.t_inter_ms if topo.nodes > 1 else topo.t_intra_ms
    steps = [max(c, link) for c in step_comp_ms[:-1]] + [float(step_comp_ms[-1])]
    return {"steps_ms": steps, "total_ms": sum(steps), "comm_bound_steps": sum(1 for c in step_comp_ms[:-1]
                                                                               if link > c), "W": W}


def hierarchical_ring_ms(step_comp_ms: Sequence[float], topo: RingTopology) -> dict:
    """Hierarchical ring: inner steps bounded by max(T_comp, T_intra); each
    round of gpus_per_node inner steps followed by another round waits for
    the outer transfer (T_inter) if the round is shorter."""
    g = topo.gpus_per_node
    steps = [max(c, topo.t_intra_ms) for c in step_comp_ms]
    rounds = [steps[i:i + g] for i in range(0, len(steps), g)]
    total, exposed = 0.0, 0.0
    for k, rd in enumerate(rounds):
        t = sum(rd)
        if k + 1 < len(rounds) and topo.nodes > 1 and topo.t_inter_ms > t:
            exposed += topo.t_inter_ms - t
            t = topo.t_inter_ms
        total += t
    return {"steps_ms": steps, "total_ms": total, "exposed_outer_ms": exposed, "W": len(steps)}


def forward_latency_ms(step_comp_ms: Sequence[float], topo: RingTopology, index_ms: float = 0.0,
                       other_ms: float = 0.0) -> dict:
    """The pages' forward-attention breakdown: index build + other (host)
    work + the ring, for both schedules, and the saving of the hierarchy."""
    f = flat_ring_ms(step_comp_ms, topo)
    h = hierarchical_ring_ms(step_comp_ms, topo)
    tf = index_ms + other_ms + f["total_ms"]
    th = index_ms + other_ms + h["total_ms"]
    return {"flat_ms": tf, "hierarchical_ms": th, "reduction": 1.0 - th / tf if tf > 0 else 0.0,
            "flat": f, "hierarchical": h}
