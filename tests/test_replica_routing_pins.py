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


# ---------------------------------------------------------------- hand-worked slots
# Expected slots below were worked out by hand from the rule's text, not
# computed with the oracle's formulas, so that a plausible misreading of the
# rule (the assignment index instead of the token index, copies in
# descending rank order, an off-by-one in the modulus, the source rank
# instead of the token) fails them.

def _slot_ranks(pl, slot):
    return [int(pl.slot_rank[int(s)]) for s in slot]


def test_fixed_rule_fallback_takes_copy_t_mod_n_in_ascending_rank_order():
    """Replica workload rule: a token on a node without a copy takes copy
    (t mod n_copies), copies in ascending rank order; otherwise the copy on
    its own node.  4 nodes of 1 rank; expert 0 has copies on ranks 3, 1, 2
    (listed out of order on purpose), expert 1 lives on rank 0.  Token t
    lives on rank t mod 4."""
    pl = wl.placement_from_hosts(2, 4, 1, [[3, 1, 2], [0]])
    T = 12
    ids = np.array([[0, 1]] * T, dtype=np.int32)
    lay = oracle.dispatch_layout(ids, pl)
    got = _slot_ranks(pl, lay["slot"][0::2])         # expert 0 is j = 0
    # node 0 tokens (t = 0, 4, 8) have no copy: t mod 3 = 0, 1, 2 -> ranks 1, 2, 3;
    # node 1/2/3 tokens keep their own node's copy
    assert got == [1, 1, 2, 3,
                   2, 1, 2, 3,
                   3, 1, 2, 3]
    assert _slot_ranks(pl, lay["slot"][1::2]) == [0] * T


def test_fixed_rule_fallback_uses_the_token_index_not_the_assignment_index():
    """k = 3 with the replicated expert last (j = 2), every token on rank 0
    (node 0, no copy there): token t takes copy t mod 3 -> ranks 1, 2, 3, 1,
    2, 3.  The assignment index a = 3t + 2 would give copy (3t + 2) mod 3 =
    2 every time."""
    src = np.zeros(6, dtype=np.int32)
    pl = wl.placement_from_hosts(3, 4, 1, [[3, 1, 2], [0], [0]], token_src_rank=src)
    ids = np.array([[1, 2, 0]] * 6, dtype=np.int32)
    lay = oracle.dispatch_layout(ids, pl)
    assert _slot_ranks(pl, lay["slot"][2::3]) == [1, 2, 3, 1, 2, 3]


def test_waterfill_two_sources_hand_worked():
    """"Zepp" Section 5, "Routing", worked by hand.  6 ranks, 2 per node
    (nodes {0,1}, {2,3}, {4,5}); expert 0 has copies p0 on rank 1 (node 0),
    p1 on rank 2 (node 1), p2 on rank 4 (node 2).  Tokens 0,2,4,6,8,9 live
    on rank 0 (demand 6), tokens 1,3,5,7 on rank 5 (demand 4); C = 1/3.

    D = 10, q = (4, 3, 3), slack = floor(10 / 9) = 1, lo = (3, 2, 2),
    hi = (5, 4, 4).
    Own-GPU pass: neither source hosts a copy.
    Own-node pass: rank 0 -> p0, allowed min(5, 10 - (2 + 2)) = 5, gives 5;
                   rank 5 -> p2, allowed min(4, 5 - (0 + 2)) = 3 (the
                   reserve for p1's lower bound binds), gives 3.
    Remote pass:   rank 0 -> p1 (p0 is on its node), allowed
                   min(4, 2 - 0) = 2, gives its last 1;
                   rank 5 -> p0 allowed min(0, ..) = 0; p1 allowed
                   min(3, 1 - 0) = 1, gives its last 1.
    Loads (5, 2, 3) lie within the bounds.
    Each source's assignments in ascending order take its destinations in
    locality order: rank 0's first five tokens (0, 2, 4, 6, 8) take p0 and
    token 9 takes p1; rank 5's first three (1, 3, 5) take p2 and token 7
    takes p1.  Tokens 7 and 9 cross nodes."""
    src = np.array([0, 5, 0, 5, 0, 5, 0, 5, 0, 0], dtype=np.int32)
    pl = wl.placement_from_hosts(1, 6, 2, [[1, 2, 4]], token_src_rank=src)
    ids = np.zeros((10, 1), dtype=np.int32)
    alloc, load, lo, hi = oracle.waterfill_expert({0: 6, 5: 4}, [1, 2, 4], 2, 1, 3)
    assert (lo, hi, load) == ([3, 2, 2], [5, 4, 4], [5, 2, 3])
    assert alloc[0] == [(0, 5), (1, 1)] and alloc[5] == [(2, 3), (1, 1)]
    slot, inter = oracle.route_replicas_waterfill(ids, pl, 1, 3)
    assert _slot_ranks(pl, slot) == [1, 4, 1, 4, 1, 4, 1, 2, 1, 2]
    assert inter == 2


# ---------------------------------------------------------------- refinement
# "Zepp", Section 5 "Routing": after water-filling, a greedy refinement
# consolidates each token's remote requests onto fewer nodes within the
# same load bounds.  The cases below are worked by hand; 4 nodes of one rank
# each, every token on rank 0 (node 0), C = 0 (exact balance).

def _refine_case(hosts, ids):
    ids = np.asarray(ids, dtype=np.int32)
    src = np.zeros(ids.shape[0], dtype=np.int32)
    pl = wl.placement_from_hosts(len(hosts), 4, 1, hosts, token_src_rank=src)
    slot, inter = oracle.route_replicas_waterfill(ids, pl, 0, 1)
    ref, before, after = oracle.refine_consolidate(ids, slot, pl)
    return pl, slot, inter, ref, before, after


def test_refinement_strictly_lowers_the_node_pairs():
    """Expert 0 on ranks 1, 2; expert 1 on ranks 2, 3; expert 2 on rank 0.
    Tokens: t0 = (0, 1), t1 = (0, 2), t2 = (2, 1).  Water-filling (C = 0)
    gives each copy of experts 0 and 1 one assignment; in ascending order
    t0 takes expert 0 on rank 1 and t1 on rank 2; t0 takes expert 1 on
    rank 2 and t2 on rank 3.  So t0 sends to nodes {1, 2}: 4 (token,
    remote node) pairs in all.  Refined: t0's two requests can both go to
    node 2 (covers 2), leaving expert 0's rank-1 copy to t1 and expert 1's
    rank-3 copy to t2: 3 pairs, the same loads, the same 4 remote
    assignments."""
    pl, slot, inter, ref, before, after = _refine_case(
        [[1, 2], [2, 3], [0]], [[0, 1], [0, 2], [2, 1]])
    assert _slot_ranks(pl, slot) == [1, 2, 2, 0, 0, 3]
    assert _slot_ranks(pl, ref) == [2, 2, 1, 0, 0, 3]
    assert (before, after, inter) == (4, 3, 4)
    assert oracle.dispatch_messages(ref, pl, 3, 2) == (4, 3)
    assert np.array_equal(np.bincount(ref, minlength=pl.n_slots),
                          np.bincount(slot, minlength=pl.n_slots))


def test_refinement_ties_go_to_the_lower_node():
    """Experts 0 and 1 both on ranks 1 and 2.  t0 = (0, 1) can put both on
    node 1 or both on node 2 (cover 2 each): the lower node, 1, wins; t1
    and t2 then take the rank-2 copies."""
    pl, slot, inter, ref, before, after = _refine_case(
        [[1, 2], [1, 2], [0]], [[0, 1], [0, 2], [2, 1]])
    assert _slot_ranks(pl, ref) == [1, 1, 2, 0, 0, 2]
    assert (before, after) == (3, 3)


def test_refinement_prefers_a_node_the_token_already_sends_to():
    """Expert 3 lives on rank 3 only; expert 0 on ranks 1 and 3.  t0 =
    (3, 0) already sends to node 3 for expert 3, so its expert-0 request
    joins it there (cover 1 on node 1 and on node 3, but node 3 is already
    used); t1 = (0, 2) takes the rank-1 copy.  The water-filling's order
    had given t0 rank 1 (2 nodes) and t1 rank 3: 3 pairs before, 2 after."""
    pl, slot, inter, ref, before, after = _refine_case(
        [[1, 3], [0], [0], [3]], [[3, 0], [0, 2]])
    assert _slot_ranks(pl, slot) == [3, 1, 3, 0]
    assert _slot_ranks(pl, ref) == [3, 3, 1, 0]
    assert (before, after) == (3, 2)


def test_refinement_keeps_local_choices_and_loads():
    """A copy on the token's node is never traded away: expert 0 on ranks 0
    and 1 (ranks 0 and 1 form node 0 here, 2 ranks per node), tokens on
    rank 0 keep rank 0 as long as the water-filling gave it."""
    src = np.zeros(4, dtype=np.int32)
    pl = wl.placement_from_hosts(3, 4, 2, [[0, 2], [3], [0]], token_src_rank=src)
    ids = np.array([[0, 1], [0, 2], [0, 1], [0, 2]], dtype=np.int32)
    slot, inter = oracle.route_replicas_waterfill(ids, pl, 0, 1)
    ref, before, after = oracle.refine_consolidate(ids, slot, pl)
    # C = 0: two assignments per copy of expert 0; tokens 0 and 1 keep rank 0
    assert _slot_ranks(pl, slot)[0::2] == [0, 0, 2, 2]
    assert _slot_ranks(pl, ref)[0::2] == [0, 0, 2, 2]
    assert np.array_equal(np.bincount(ref, minlength=pl.n_slots),
                          np.bincount(slot, minlength=pl.n_slots))


def _brute_min_pairs(ids, slot, pl, i):
    """Fewest (token, remote node) pairs for source i over every way to give
    its re-choosable requests (replicated expert, remote copy in the input)
    remote copies with the input's per-copy counts."""
    T, k = ids.shape
    rpn = pl.ranks_per_node
    src = pl.token_src_rank
    n_i = i // rpn
    reps = lambda e: [int(s) for s in pl.rep_slots[pl.rep_offsets[e]:pl.rep_offsets[e + 1]]]
    free = [a for a in range(T * k) if src[a // k] == i and len(reps(int(ids.flat[a]))) > 1
            and int(pl.slot_rank[slot[a]]) // rpn != n_i]
    need = {}
    for a in free:
        need[int(slot[a])] = need.get(int(slot[a]), 0) + 1
    options = [[s for s in reps(int(ids.flat[a])) if int(pl.slot_rank[s]) // rpn != n_i]
               for a in free]
    best = None
    for choice in itertools.product(*options):
        cnt = {}
        for s in choice:
            cnt[s] = cnt.get(s, 0) + 1
        if cnt != need:
            continue
        sl = slot.copy()
        sl[free] = choice
        p = sum(len({int(pl.slot_rank[sl[t * k + j]]) // rpn for j in range(k)} - {n_i})
                for t in range(T) if src[t] == i)
        best = p if best is None else min(best, p)
    return best


@pytest.mark.parametrize("seed", range(30))
def test_refinement_against_brute_force(seed):
    """Tiny random instances: the refined routing keeps every copy's load
    and every source's per-copy counts (so the load bounds of Eq. 1 hold as
    before), never raises the (token, remote node) pairs, and is never
    below the brute-force optimum under those counts."""
    rng = np.random.default_rng(500 + seed)
    R, rpn, E, k = 4, 1, 4, 2
    T = int(rng.integers(2, 6))
    hosts = [sorted(rng.choice(R, size=int(rng.integers(1, 4)), replace=False).tolist())
             for _ in range(E)]
    src = rng.integers(0, 2, size=T).astype(np.int32)
    pl = wl.placement_from_hosts(E, R, rpn, hosts, token_src_rank=src)
    ids = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)], dtype=np.int32)
    c = (int(rng.integers(0, 3)), 2)
    slot, inter = oracle.route_replicas_waterfill(ids, pl, *c)
    ref, before, after = oracle.refine_consolidate(ids, slot, pl)
    assert np.array_equal(pl.slot_expert[ref], ids.reshape(-1))
    assert np.array_equal(np.bincount(ref, minlength=pl.n_slots),
                          np.bincount(slot, minlength=pl.n_slots))
    for i in range(R):
        for s in range(pl.n_slots):
            mine = [a for a in range(T * k) if src[a // k] == i]
            assert sum(ref[a] == s for a in mine) == sum(slot[a] == s for a in mine)
    assert oracle.dispatch_messages(slot, pl, T, k) == (inter, before)
    assert oracle.dispatch_messages(ref, pl, T, k) == (inter, after)
    assert after <= before
    assert after >= sum(_brute_min_pairs(ids, slot, pl, i) or 0 for i in range(R))
