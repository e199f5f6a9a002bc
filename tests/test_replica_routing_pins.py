"""Pins of the oracle's locality-preferred replica routing ("Zepp",
Section 4.1, Eq. 1, and Section 5 "Routing") to facts outside itself:
the constraints of Eq. 1, the Figure 6 scenario, closed forms, and brute
force over every integer routing of tiny instances.  CPU only."""

import itertools

import numpy as np
import pytest

import oracle
import workloads as wl


def _check_feasible(demand, rep_ranks, c, alloc, load, lo, hi):
    D = sum(demand.values())
    n = len(rep_ranks)
    M = {i: [0] * n for i in demand}
    for i, lst in alloc.items():
        for p, x in lst:
            assert x > 0
            M[i][p] += x
    for i in demand:                                   # row totals (Eq. 1, first constraint)
        assert sum(M[i]) == demand[i]
    for p in range(n):                                 # integer load bounds
        assert sum(M[i][p] for i in demand) == load[p]
        assert lo[p] <= load[p] <= hi[p]
    q = D / n
    slack = np.floor(c * D / n)
    for p in range(n):                                 # |load - q| <= C q, up to rounding
        assert abs(load[p] - q) <= slack + 1
    return M


@pytest.mark.parametrize("seed", range(60))
def test_waterfill_is_feasible(seed):
    rng = np.random.default_rng(seed)
    R, rpn = int(rng.choice([4, 8, 16])), int(rng.choice([1, 2, 4]))
    n = int(rng.integers(2, min(R, 5) + 1))
    rep_ranks = sorted(rng.choice(R, size=n, replace=False).tolist())
    demand = {i: int(v) for i, v in enumerate(rng.integers(0, 40, size=R)) if v > 0}
    if not demand:
        demand = {0: 1}
    c_num, c_den = int(rng.integers(0, 4)), int(rng.choice([1, 2, 10]))
    alloc, load, lo, hi = oracle.waterfill_expert(demand, rep_ranks, rpn, c_num, c_den)
    _check_feasible(demand, rep_ranks, c_num / c_den, alloc, load, lo, hi)


def test_zero_relaxation_gives_exact_balance():
    demand = {0: 30, 1: 0, 2: 3, 5: 27}
    alloc, load, lo, hi = oracle.waterfill_expert(demand, [1, 4, 6], 2, 0, 1)
    assert load == [20, 20, 20] and lo == hi == [20, 20, 20]


def test_reserve_keeps_lower_bounds_reachable():
    # Rank 0 alone could fill its local replica to the upper bound; the
    # reserve rule must leave enough for the remote replica's lower bound.
    demand = {0: 10}
    alloc, load, lo, hi = oracle.waterfill_expert(demand, [0, 4], 4, 1, 5)   # C = 0.2
    assert lo == [4, 4] and hi == [6, 6]
    assert load == [6, 4]
    assert alloc[0] == [(0, 6), (1, 4)]


def test_figure6_full_coverage_stays_local_partial_goes_remote():
    """"Zepp" Figure 6: E0 replicated on every node is served locally; E1,
    replicated on all nodes but one, sends only that node's tokens across
    nodes."""
    R, rpn = 8, 2                                     # 4 nodes of 2 GPUs
    hosts = [[0, 2, 4, 6], [1, 3, 5]]                 # E0 on every node, E1 not on node 3
    src = np.arange(16) % R
    pl = wl.placement_from_hosts(2, R, rpn, hosts, token_src_rank=np.concatenate([src, src]))
    ids = np.concatenate([np.zeros(16, np.int32), np.ones(16, np.int32)])[:, None]
    slot, inter = oracle.route_replicas_waterfill(ids, pl, 1, 1)   # C = 1: loose bounds
    node = lambda r: r // rpn
    for a in range(32):
        same = node(int(pl.slot_rank[slot[a]])) == node(int(pl.token_src_rank[a]))
        if ids[a, 0] == 0:
            assert same
        else:
            assert same == (node(int(pl.token_src_rank[a])) != 3)
    assert inter == 4                                  # E1's tokens from node 3 (ranks 6, 7), twice


def _brute_min_remote(demand, rep_ranks, rpn, lo, hi):
    """Fewest inter-node assignments over every integer routing meeting the
    row totals and the load bounds (Eq. 1 with a_ij = 1 across nodes, 0
    within a node)."""
    srcs = sorted(demand)
    n = len(rep_ranks)
    best = None

    def splits(total, parts):
        if parts == 1:
            yield (total,)
            return
        for x in range(total + 1):
            for rest in splits(total - x, parts - 1):
                yield (x,) + rest

    for rows in itertools.product(*[list(splits(demand[i], n)) for i in srcs]):
        loads = [sum(r[p] for r in rows) for p in range(n)]
        if all(lo[p] <= loads[p] <= hi[p] for p in range(n)):
            cost = sum(r[p] for i, r in zip(srcs, rows) for p in range(n)
                       if rep_ranks[p] // rpn != i // rpn)
            best = cost if best is None else min(best, cost)
    return best


@pytest.mark.parametrize("seed", range(25))
def test_waterfill_against_brute_force_optimum(seed):
    rng = np.random.default_rng(100 + seed)
    R, rpn = 4, 2
    n = int(rng.integers(2, 4))
    rep_ranks = sorted(rng.choice(R, size=n, replace=False).tolist())
    demand = {i: int(v) for i, v in enumerate(rng.integers(0, 5, size=R)) if v > 0} or {0: 2}
    c_num, c_den = int(rng.integers(0, 3)), 2
    alloc, load, lo, hi = oracle.waterfill_expert(demand, rep_ranks, rpn, c_num, c_den)
    M = _check_feasible(demand, rep_ranks, c_num / c_den, alloc, load, lo, hi)
    greedy = sum(M[i][p] for i in M for p in range(n) if rep_ranks[p] // rpn != i // rpn)
    opt = _brute_min_remote(demand, rep_ranks, rpn, lo, hi)
    assert opt is not None and greedy >= opt
    # with no lower bounds to reserve for and every node's demand within its
    # own replicas' capacity, nothing needs to leave its node
    node_cap = {}
    for p, r in enumerate(rep_ranks):
        node_cap[r // rpn] = node_cap.get(r // rpn, 0) + hi[p]
    node_dem = {}
    for i, d in demand.items():
        node_dem[i // rpn] = node_dem.get(i // rpn, 0) + d
    if all(x == 0 for x in lo) and all(d <= node_cap.get(nd, 0) for nd, d in node_dem.items()):
        assert greedy == opt == 0


def test_route_replicas_assigns_every_assignment_to_a_copy_of_its_expert():
    w = wl.WORKLOADS["replica"].scaled(T=1024)
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    for c in [(0, 1), (1, 10), (1, 1)]:
        slot, inter = oracle.route_replicas_waterfill(ids, pl, *c)
        assert np.array_equal(pl.slot_expert[slot], ids.reshape(-1))
        lay = oracle.dispatch_layout_from_slots(ids, slot, pl)
        assert lay["seg_counts"].sum() == w.A
