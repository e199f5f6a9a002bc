"""Pins of the oracle's simulated merge ("Zepp", Section 3.2 "Redundant
Tokens" and Section 4.2 "Merge"; Algorithm 1's PreReduce / Reduce): the
Figure 4 case, an independent count of token/node pairs, and reductions
of the pre-reduced combine to the plain combine.  CPU only."""

import numpy as np

import oracle
import workloads as wl


def test_figure4_shared_remote_node_crosses_once():
    # two nodes of one rank; the token lives on rank 0 and picks two experts
    # hosted on node 1 and one on its own node
    pl = wl.placement_from_hosts(3, 2, 1, [[1], [1], [0]], token_src_rank=np.array([0]))
    ids = np.array([[0, 1, 2]], np.int32)
    slot = np.array([oracle.choose_slot(int(e), 0, pl) for e in ids[0]], np.int32)
    assert oracle.dispatch_messages(slot, pl, 1, 3) == (2, 1)


def test_dispatch_message_counts_against_independent_count():
    w = wl.WORKLOADS["replica"].scaled(T=2048)
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = oracle.dispatch_layout(ids, pl)
    before, after = oracle.dispatch_messages(lay["slot"], pl, w.T, w.k)
    t = np.arange(w.A) // w.k
    src_node = (t % w.R) // w.ranks_per_node
    dst_node = pl.slot_rank[lay["slot"]] // w.ranks_per_node
    remote = dst_node != src_node
    assert before == int(remote.sum())
    assert after == len(np.unique(t[remote] * 1000 + dst_node[remote]))
    assert after <= before


def _bits(x):
    return oracle.f64_to_bf16_bits(oracle.bf16_round(x))


def test_pre_reduction_on_one_node_is_the_plain_combine():
    rng = np.random.default_rng(3)
    T, k, H = 50, 4, 64
    yp = _bits(rng.standard_normal((T * k, H)))
    dr = rng.permutation(T * k).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    one_node = np.zeros(T * k, np.int32)
    assert np.array_equal(oracle.combine_merged_fma32(yp, dr, w, one_node),
                          oracle.combine_fma32(yp, dr, w))


def test_pre_reduction_differs_from_plain_only_by_the_partial_rounding():
    rng = np.random.default_rng(4)
    T, k, H = 60, 8, 96
    yp = _bits(rng.standard_normal((T * k, H)))
    sh = _bits(rng.standard_normal((T, H)))
    dr = rng.permutation(T * k).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    node = rng.integers(0, 4, T * k).astype(np.int32)
    f = oracle.bf16_bits_to_f64
    merged32 = f(oracle.combine_merged_fma32(yp, dr, w, node, sh))
    merged64 = oracle.combine_merged_f64(f(yp), dr, w.astype(np.float64), node, f(sh))
    plain64 = oracle.combine_f64(f(yp), dr, w.astype(np.float64), f(sh))
    # fp32 fma chains vs fp64 sums of the same definition: at most a few ulps
    assert np.max(np.abs(merged32 - merged64) / (np.abs(merged64) + 1e-3)) < 3e-2
    assert np.linalg.norm(merged32 - merged64) / np.linalg.norm(merged64) < 1e-2
    # each bf16-rounded partial moves the sum by at most half an ulp of itself
    ulp = lambda v: np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 1e-30))[1] - 8)
    bound = np.zeros_like(plain64)
    for t in range(T):
        for n in set(node[t * k:(t + 1) * k].tolist()):
            part = sum(float(w[t, j]) * f(yp)[dr[t * k + j]] for j in range(k)
                       if node[t * k + j] == n)
            bound[t] += ulp(part) / 2
    assert np.all(np.abs(merged64 - plain64) <= bound + ulp(plain64) + ulp(merged64))
