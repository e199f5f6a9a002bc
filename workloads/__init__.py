"""Seeded synthetic inputs for the MoE-layer hot path.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It holds only input generation: shapes, seeds, value
distributions and expert placements.  None of the layer's arithmetic
(routing, layout, permutation, expert FFN, combine, balancedness) lives here.

Workloads (sizes follow the shapes the pages use):
  tiny          8 tokens, hidden 256, 64 experts, top-2, I=128, 8 ranks
                (the 8-token / 64-expert / top-2 example of "Serving
                Mixture-of-Experts Models", "Follow one token through an MoE
                layer").
  decode        64 tokens, hidden 8192, 64 experts, top-2, I=2048, 8 ranks
                ("Price one dispatch": 64 decode sequences, 16 KiB rows).
  prefill       4000 tokens, same layer ("Price one dispatch": a 4,000-token
                prompt).
  group_limited 4096 tokens, hidden 7168, 256 experts in 8 groups, top-4
                groups by the sum of each group's top-2 sigmoid scores, then
                top-8 experts, I=2048, plus one shared expert (I=2048), 32
                ranks ("Mixture-of-Experts Inference", "MoE architecture
                recap": grouped routed experts and shared experts).
  replica       16384 tokens, hidden 4096, 32 experts, top-4, I=1536, 16
                ranks in 4 nodes of 4; the 4 hottest experts get 2 extra
                replicas on distinct nodes ("Zepp", Section 4.1 "Expert
                replication and placement").

Value distributions: router logits fp32 ~ N(0,1) plus a per-expert Zipf bias
-s*ln(rank) over a seeded random expert order; activations bf16 ~ N(0,1);
weights bf16 ~ N(0, 0.02).  Floating values are drawn in fp32 by torch's
seeded generator on the requested device and rounded to bf16
(round-to-nearest-even).  The same arrays feed both the CUDA path and the
oracle within one run; the draw itself depends on the device, so a run never
mixes a CPU draw with a GPU draw.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed namespace
    T: int                # tokens
    H: int                # hidden width
    E: int                # routed experts
    k: int                # experts per token
    I: int                # expert FFN intermediate width
    R: int                # simulated EP ranks
    ranks_per_node: int
    score_fn: int = SCORE_SOFTMAX
    n_groups: int = 1
    topk_groups: int = 1
    group_topn: int = 1
    shared_I: int = 0     # 0 = no shared expert
    zipf_s: float = 0.0
    hot_experts: int = 0  # experts that get extra replicas
    extra_replicas: int = 0

    @property
    def A(self) -> int:
        """Assignments: every token is routed to k experts."""
        return self.T * self.k

    def with_zipf(self, s: float) -> "Workload":
        return dataclasses.replace(self, zipf_s=float(s))

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, T=8, H=256, E=64, k=2, I=128, R=8, ranks_per_node=8),
    "decode": Workload("decode", 2, T=64, H=8192, E=64, k=2, I=2048, R=8,
                       ranks_per_node=8, zipf_s=1.0),
    "prefill": Workload("prefill", 3, T=4000, H=8192, E=64, k=2, I=2048, R=8,
                        ranks_per_node=8, zipf_s=1.0),
    "group_limited": Workload("group_limited", 4, T=4096, H=7168, E=256, k=8,
                              I=2048, R=32, ranks_per_node=8,
                              score_fn=SCORE_SIGMOID, n_groups=8, topk_groups=4,
                              group_topn=2, shared_I=2048, zipf_s=0.8),
    "replica": Workload("replica", 5, T=16384, H=4096, E=32, k=4, I=1536, R=16,
                        ranks_per_node=4, zipf_s=1.0, hot_experts=4,
                        extra_replicas=2),
}

REPLICA_ZIPF_SWEEP = (0.0, 0.5, 1.0, 1.5)

# tensor ids inside a workload's seed namespace
_T_LOGITS, _T_ZIPF_ORDER, _T_X, _T_WGU, _T_WD, _T_SWGU, _T_SWD = range(1, 8)


def seed_for(w: Workload, tensor_id: int) -> int:
    return 1000 * w.index + tensor_id


# ---------------------------------------------------------------- placement
@dataclasses.dataclass
class Placement:
    """Physical expert slots, one per (rank, expert) pair that hosts weights.

    slot_expert / slot_rank are sorted by (rank, expert); segment s of the
    dispatched buffer belongs to slot s.  rep_offsets / rep_slots list, for
    each expert, its slots in ascending rank order (CSR).  token_src_rank
    (optional) names the rank each token lives on; None means t mod R.
    """
    n_experts: int
    n_ranks: int
    ranks_per_node: int
    slot_expert: np.ndarray
    slot_rank: np.ndarray
    rep_offsets: np.ndarray
    rep_slots: np.ndarray
    token_src_rank: Optional[np.ndarray] = None

    @property
    def n_slots(self) -> int:
        return int(self.slot_expert.shape[0])


def placement_from_hosts(n_experts: int, n_ranks: int, ranks_per_node: int,
                         hosts: List[List[int]],
                         token_src_rank: Optional[np.ndarray] = None) -> Placement:
    """hosts[e] = list of ranks holding a copy of expert e."""
    pairs = sorted((r, e) for e in range(n_experts) for r in set(hosts[e]))
    slot_expert = np.array([e for r, e in pairs], dtype=np.int32)
    slot_rank = np.array([r for r, e in pairs], dtype=np.int32)
    rep_offsets = np.zeros(n_experts + 1, dtype=np.int32)
    rep_lists = [[] for _ in range(n_experts)]
    for s, (r, e) in enumerate(pairs):
        rep_lists[e].append(s)
    for e in range(n_experts):
        rep_lists[e].sort(key=lambda s: int(slot_rank[s]))
        rep_offsets[e + 1] = rep_offsets[e] + len(rep_lists[e])
    rep_slots = np.array([s for lst in rep_lists for s in lst], dtype=np.int32)
    return Placement(n_experts, n_ranks, ranks_per_node, slot_expert, slot_rank,
                     rep_offsets, rep_slots,
                     None if token_src_rank is None else np.asarray(token_src_rank, np.int32))


def round_robin_hosts(n_experts: int, n_ranks: int) -> List[List[int]]:
    """Expert e lives on rank e mod R (the round-robin mapping of "Zepp",
    Figure 1)."""
    return [[e % n_ranks] for e in range(n_experts)]


def zipf_order(w: Workload) -> np.ndarray:
    """Seeded random expert order; position p (0-based) has Zipf rank p+1."""
    rng = np.random.default_rng(seed_for(w, _T_ZIPF_ORDER))
    return rng.permutation(w.E).astype(np.int64)


def zipf_bias(w: Workload) -> np.ndarray:
    """Per-expert logit bias log(1/rank^s) = -s*ln(rank), fp32."""
    order = zipf_order(w)
    rank = np.empty(w.E, dtype=np.float64)
    rank[order] = np.arange(1, w.E + 1, dtype=np.float64)
    return (-w.zipf_s * np.log(rank)).astype(np.float32)


def replica_hosts(w: Workload) -> List[List[int]]:
    """Round-robin base placement plus extra replicas for the hottest experts.

    The hottest experts are Zipf ranks 1..hot_experts of the seeded order
    (the same experts at every Zipf exponent).  Following the hierarchical
    rule of "Zepp" Section 4.1 (replicas spread round-robin across nodes,
    then within a node to the least-loaded GPU), expert e with home node n0
    gets its extra replicas on nodes n0+1, n0+2, ... (mod nodes); inside a
    node the rank with the fewest slots so far is used (ties: lowest rank).
    """
    hosts = round_robin_hosts(w.E, w.R)
    n_nodes = w.R // w.ranks_per_node
    slots_on = [0] * w.R
    for e in range(w.E):
        for r in hosts[e]:
            slots_on[r] += 1
    for e in [int(v) for v in zipf_order(w)[: w.hot_experts]]:
        n0 = hosts[e][0] // w.ranks_per_node
        for i in range(1, w.extra_replicas + 1):
            node = (n0 + i) % n_nodes
            ranks = range(node * w.ranks_per_node, (node + 1) * w.ranks_per_node)
            r = min(ranks, key=lambda rr: (slots_on[rr], rr))
            hosts[e].append(r)
            slots_on[r] += 1
    return hosts


def make_placement(w: Workload) -> Placement:
    if w.hot_experts > 0:
        hosts = replica_hosts(w)
    else:
        hosts = round_robin_hosts(w.E, w.R)
    return placement_from_hosts(w.E, w.R, w.ranks_per_node, hosts)


# ---------------------------------------------------------------- tensors
def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_logits(w: Workload, device="cpu") -> torch.Tensor:
    g = _gen(device, seed_for(w, _T_LOGITS))
    logits = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32)
    if w.zipf_s != 0.0:
        logits += torch.from_numpy(zipf_bias(w)).to(device)[None, :]
    return logits


def make_x(w: Workload, device="cpu") -> torch.Tensor:
    g = _gen(device, seed_for(w, _T_X))
    return torch.randn(w.T, w.H, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def _weights(n: int, rows: int, cols: int, seed: int, device) -> torch.Tensor:
    """bf16 ~ N(0, 0.02) of shape [n, rows, cols], drawn one matrix at a time
    so that the fp32 temporary stays small."""
    g = _gen(device, seed)
    out = torch.empty(n, rows, cols, dtype=torch.bfloat16, device=device)
    for i in range(n):
        tmp = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
        tmp.mul_(0.02)
        out[i].copy_(tmp)
    return out


def make_w_gate_up(w: Workload, device="cpu") -> torch.Tensor:
    """[E, 2I, H]: rows 0..I-1 are the gate projection, rows I..2I-1 the up
    projection, each row a K-major (H-contiguous) vector."""
    return _weights(w.E, 2 * w.I, w.H, seed_for(w, _T_WGU), device)


def make_w_down(w: Workload, device="cpu") -> torch.Tensor:
    """[E, H, I]: row h is the I-contiguous vector producing output column h."""
    return _weights(w.E, w.H, w.I, seed_for(w, _T_WD), device)


def make_shared_weights(w: Workload, device="cpu"):
    if w.shared_I == 0:
        return None, None
    gu = _weights(1, 2 * w.shared_I, w.H, seed_for(w, _T_SWGU), device)
    d = _weights(1, w.H, w.shared_I, seed_for(w, _T_SWD), device)
    return gu, d


def bytes_per_row(w: Workload) -> int:
    """bf16 bytes of one routed activation row."""
    return 2 * w.H


def small_parity_workload(name: str = "parity_small", **kw) -> Workload:
    """A layer small enough for the oracle to finish in seconds that still
    spans several 128-row tiles per expert, ragged tails, and several output
    column tiles."""
    base = dict(index=90, T=300, H=512, E=8, k=2, I=384, R=4, ranks_per_node=2,
                zipf_s=0.7)
    base.update(kw)
    return Workload(name, **base)
