"""Pins of the CPU oracle to facts outside itself: the pages' worked
examples (tests/golden), brute force on tiny inputs, closed forms, and
special cases that reduce to a library routine.  CPU only."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def brute_topk(scores, k):
    """The unique k-subset whose members each beat every non-member (beat =
    higher score, or equal score and lower index), ordered by that relation.
    Exponential enumeration; tiny inputs only."""
    n = len(scores)

    def beats(a, b):
        return scores[a] > scores[b] or (scores[a] == scores[b] and a < b)

    found = [sub for sub in itertools.combinations(range(n), k)
             if all(beats(a, b) for a in sub for b in range(n) if b not in sub)]
    assert len(found) == 1
    rest, ordered = list(found[0]), []
    while rest:
        best = rest[0]
        for m in rest[1:]:
            if beats(m, best):
                best = m
        ordered.append(best)
        rest.remove(best)
    return ordered


# ------------------------------------------------------------------ bf16
def test_bf16_round_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # exact ties between two bf16 neighbours, both parities
    base = rng.standard_normal(1000).astype(np.float32)
    bits = (base.view(np.uint32) & 0xFFFF0000) | 0x00008000
    v = np.concatenate([v, bits.view(np.float32), (bits + 0x10000).view(np.float32)])
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_no_double_rounding():
    # 1 + 2^-8 is a tie between bf16 1.0 and 1.0078125; anything above must go up.
    # fp32 would first round 1 + 2^-8 + 2^-40 to the tie and then down to even.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_round(x) == 1.0 + 2.0 ** -7
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 1.0          # tie -> even
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2 * 2.0 ** -7  # tie -> even (up)


# ------------------------------------------------------------------ routers
def _tiny_logit_cases(seed, n, E_max=8, values=(-1.0, -0.0, 0.0, 0.5, 1.0, 2.0)):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        E = int(rng.integers(2, E_max + 1))
        k = int(rng.integers(1, min(3, E) + 1))
        row = rng.choice(np.array(values, dtype=np.float32), size=E)
        yield E, k, row


def test_softmax_topk_matches_brute_force_with_ties():
    for E, k, row in _tiny_logit_cases(1, 400):
        ids, w = oracle.route_softmax_topk(row[None, :], k)
        want = brute_topk([float(v) for v in row], k)
        assert list(ids[0]) == want, (row, k)
        p = scipy.special.softmax(row.astype(np.float64))
        np.testing.assert_allclose(w[0], p[want] / p[want].sum(), rtol=1e-14)


def test_softmax_weights_closed_forms():
    # two experts whose logits differ by ln 3 -> 3/4 and 1/4
    ids, w = oracle.route_softmax_topk(np.array([[0.0, math.log(3.0), -5.0]], np.float32), 2)
    assert list(ids[0]) == [1, 0]
    d = float(np.float32(math.log(3.0)))
    np.testing.assert_allclose(w[0], [math.exp(d) / (1 + math.exp(d)), 1 / (1 + math.exp(d))], rtol=1e-15)
    np.testing.assert_allclose(w[0], [0.75, 0.25], rtol=1e-7)
    # equal logits -> 1/k each, lowest ids first
    ids, w = oracle.route_softmax_topk(np.zeros((1, 6), np.float32), 4)
    assert list(ids[0]) == [0, 1, 2, 3]
    np.testing.assert_allclose(w[0], [0.25] * 4, rtol=0, atol=0)
    # k = E -> the full softmax (library routine)
    rng = np.random.default_rng(3)
    row = rng.standard_normal(16).astype(np.float32)
    ids, w = oracle.route_softmax_topk(row[None, :], 16)
    np.testing.assert_allclose(w[0], scipy.special.softmax(row.astype(np.float64))[ids[0]], rtol=1e-13)


def _brute_group_limited(row, k, n_groups, topk_groups, group_topn):
    E = len(row)
    gs = E // n_groups
    sig = scipy.special.expit(row.astype(np.float64))
    gscore = []
    for g in range(n_groups):
        members = [float(v) for v in row[g * gs:(g + 1) * gs]]
        top = brute_topk(members, group_topn)
        s = 0.0
        for i in top:
            s += sig[g * gs + i]
        gscore.append(s)
    groups = brute_topk(gscore, topk_groups)
    cand = sorted(e for g in groups for e in range(g * gs, (g + 1) * gs))
    sub = brute_topk([float(row[e]) for e in cand], k)
    chosen = [cand[i] for i in sub]
    s = sig[chosen]
    return chosen, s / s.sum()


def test_group_limited_matches_brute_force():
    rng = np.random.default_rng(7)
    vals = np.array([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 1.5, 3.0], np.float32)
    for trial in range(200):
        n_groups = int(rng.choice([2, 4]))
        gs = int(rng.choice([2, 4]))
        E = n_groups * gs
        topk_groups = int(rng.integers(1, n_groups + 1))
        group_topn = int(rng.integers(1, gs + 1))
        k = int(rng.integers(1, min(4, topk_groups * gs) + 1))
        row = rng.choice(vals, size=E) if trial % 2 else rng.standard_normal(E).astype(np.float32)
        ids, w, _ = oracle.route_group_limited(row[None, :], k, n_groups, topk_groups, group_topn)
        want, ww = _brute_group_limited(row, k, n_groups, topk_groups, group_topn)
        assert list(ids[0]) == want, (row, k, n_groups, topk_groups, group_topn)
        np.testing.assert_allclose(w[0], ww, rtol=1e-14)


def test_group_limited_with_all_groups_is_plain_sigmoid_topk():
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((20, 32)).astype(np.float32)
    ids, w, _ = oracle.route_group_limited(lg, 5, 8, 8, 2)
    for t in range(20):
        want = brute_topk([float(v) for v in lg[t]], 5)
        assert list(ids[t]) == want
        s = scipy.special.expit(lg[t].astype(np.float64))[want]
        np.testing.assert_allclose(w[t], s / s.sum(), rtol=1e-14)


def test_group_limit_excludes_experts_outside_kept_groups():
    # group 0 holds the single best expert but a weak second; group 1 two
    # strong experts: with top-1 group by top-2 sum, group 1 wins and the
    # globally best expert 0 must not be chosen.
    row = np.array([5.0, -5.0, 3.0, 3.0], np.float32)
    ids, w, _ = oracle.route_group_limited(row[None, :], 1, 2, 1, 2)
    assert list(ids[0]) == [2]
    ids, w, _ = oracle.route_group_limited(row[None, :], 1, 2, 1, 1)   # top-1 sum
    assert list(ids[0]) == [0]


# ------------------------------------------------------------------ layout
def _check_layout_invariants(topk_ids, pl, lay):
    T, k = topk_ids.shape
    A = T * k
    S = pl.n_slots
    c, o, d, sa = lay["seg_counts"], lay["seg_offsets"], lay["dest_row"], lay["src_assign"]
    assert c.sum() == A
    assert o[0] == 0 and o[-1] == A and np.all(np.diff(o) == c)
    assert np.array_equal(np.sort(d), np.arange(A))                 # bijection
    assert np.array_equal(sa[d], np.arange(A))                      # inverse
    assert np.array_equal(d[sa], np.arange(A))
    for s in range(S):
        seg = sa[o[s]:o[s + 1]]
        assert np.all(np.diff(seg) > 0)                             # stable
        assert np.all(lay["slot"][seg] == s)
    assert np.array_equal(pl.slot_expert[lay["slot"]], topk_ids.reshape(-1))   # hosts its expert
    per_rank = np.bincount(pl.slot_rank[lay["slot"]], minlength=pl.n_ranks)
    assert np.array_equal(per_rank, lay["rank_counts"])


@pytest.mark.parametrize("name", ["tiny", "replica"])
def test_layout_invariants(name):
    w = wl.WORKLOADS[name]
    if name == "replica":
        w = w.scaled(T=512)
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = oracle.dispatch_layout(ids, pl)
    _check_layout_invariants(ids, pl, lay)


def test_replica_rule_prefers_own_node_and_spreads_otherwise():
    w = wl.WORKLOADS["replica"].scaled(T=2048)
    pl = wl.make_placement(w)
    assert pl.n_slots == w.E + w.hot_experts * w.extra_replicas
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = oracle.dispatch_layout(ids, pl)
    node_of = lambda r: r // w.ranks_per_node
    spread = {}
    for a in range(w.A):
        t, e, s = a // w.k, int(ids.reshape(-1)[a]), int(lay["slot"][a])
        reps = list(pl.rep_slots[pl.rep_offsets[e]:pl.rep_offsets[e + 1]])
        assert s in reps
        own = [r for r in reps if node_of(pl.slot_rank[r]) == node_of(t % w.R)]
        if own:
            assert s == own[0]
        else:
            spread.setdefault(e, set()).add(s)
    # experts with copies on other nodes but not this one spread over all copies
    assert any(len(v) > 1 for v in spread.values())


def test_follow_one_token_counts():
    g = golden("dispatch_pricing.json")["follow_one_token"]
    w = wl.WORKLOADS["tiny"]
    assert (w.T, w.E, w.k, w.R) == (g["tokens"], g["experts"], g["k"], g["gpus"])
    ids, wts = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = oracle.dispatch_layout(ids, wl.make_placement(w))
    assert lay["seg_counts"].sum() == g["expert_executions"] == w.A
    y_perm = np.random.default_rng(0).standard_normal((w.A, 4))
    assert oracle.combine_f64(y_perm, lay["dest_row"], wts).shape[0] == g["outputs_combined_into"]
    assert round(100 * w.k / w.E) == g["expert_param_fraction_percent_roughly"]


def test_price_one_dispatch_bytes():
    g = golden("dispatch_pricing.json")["price_one_dispatch"]
    dec, pre = wl.WORKLOADS["decode"], wl.WORKLOADS["prefill"]
    assert dec.H == pre.H == g["hidden"]
    assert wl.bytes_per_row(dec) == g["bytes_per_row"]
    assert (dec.T, dec.A) == (g["decode_tokens"], g["decode_assignments"])
    assert dec.A * wl.bytes_per_row(dec) == g["decode_bytes_one_direction"]
    assert 2 * dec.A * wl.bytes_per_row(dec) == g["decode_bytes_per_layer_step"]
    assert (pre.T, pre.A) == (g["prefill_tokens"], g["prefill_assignments"])
    assert pre.A * wl.bytes_per_row(pre) == g["prefill_bytes_one_direction"]


# ------------------------------------------------------------------ balance
def _ids_with_counts(counts):
    return np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]


@pytest.mark.parametrize("case", ["contiguous_pairs", "repack", "replicate_e0_on_rank3"])
def test_worked_example_balancedness(case):
    g = golden("worked_example_balance.json")
    cs = g["cases"][case]
    ids = _ids_with_counts(g["expert_counts"])
    T = ids.shape[0]
    assert T == g["total_assignments"]
    if case == "replicate_e0_on_rank3":
        # each rank is its own node; E0's tokens alternate between the ranks
        # holding its two copies, so the split is even
        src = np.zeros(T, np.int32)
        e0 = np.nonzero(ids[:, 0] == 0)[0]
        src[e0[1::2]] = 3
        pl = wl.placement_from_hosts(8, 4, 1, cs["hosts"], token_src_rank=src)
    else:
        pl = wl.placement_from_hosts(8, 4, 4, cs["hosts"])
    lay = oracle.dispatch_layout(ids, pl)
    _check_layout_invariants(ids, pl, lay)
    assert list(lay["rank_counts"]) == cs["rank_loads"]
    bal, mx, total = oracle.balance_stats(lay["rank_counts"])
    assert total == g["total_assignments"] and mx == max(cs["rank_loads"])
    assert bal == cs["balancedness_num"] / cs["balancedness_den"]


def test_uniform_load_is_exactly_one():
    w = wl.WORKLOADS["tiny"]
    lg = np.full((w.T, w.E), -4.0, np.float32)
    for t in range(w.T):
        lg[t, t] = 2.0          # rank t mod 8
        lg[t, t + 8] = 1.0      # rank (t+8) mod 8 = t mod 8
    ids, _ = oracle.route_softmax_topk(lg, 2)
    lay = oracle.dispatch_layout(ids, wl.make_placement(w))
    assert list(lay["rank_counts"]) == [2] * 8
    assert oracle.balance_stats(lay["rank_counts"]) == (1.0, 2, 16)


def test_balance_with_nothing_routed():
    assert oracle.balance_stats(np.zeros(4, np.int32)) == (1.0, 0, 0)


# ------------------------------------------------------------------ permute / combine
def _bf16_bits(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_permute_rows_are_their_sources_and_inverse_is_identity():
    w = wl.WORKLOADS["replica"].scaled(T=256, H=64)
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = oracle.dispatch_layout(ids, pl)
    rng = np.random.default_rng(4)
    x = _bf16_bits(rng, (w.T, w.H))
    xp = oracle.permute(x, lay["dest_row"], w.k)
    for r in range(w.A):
        assert np.array_equal(xp[r], x[lay["src_assign"][r] // w.k])
    # combine with one-hot weights undoes the permutation bit for bit
    onehot = np.zeros((w.T, w.k))
    onehot[:, 0] = 1.0
    back = oracle.combine_f64(oracle.bf16_bits_to_f64(xp), lay["dest_row"], onehot)
    assert np.array_equal(oracle.f64_to_bf16_bits(back), x)
    # dyadic weights summing to one over identical copies: also exact
    quarter = np.tile(np.array([0.25, 0.25, 0.125, 0.375]), (w.T, 1))
    back = oracle.combine_f64(oracle.bf16_bits_to_f64(xp), lay["dest_row"], quarter)
    assert np.array_equal(oracle.f64_to_bf16_bits(back), x)
    back32 = oracle.combine_fma32(xp, lay["dest_row"], quarter.astype(np.float32))
    assert np.array_equal(back32, x)


def test_combine_fma32_against_fp64_and_shared_only():
    rng = np.random.default_rng(5)
    T, k, H = 40, 4, 96
    yp = _bf16_bits(rng, (T * k, H))
    sh = _bf16_bits(rng, (T, H))
    dr = rng.permutation(T * k).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    got = oracle.bf16_bits_to_f64(oracle.combine_fma32(yp, dr, w, sh))
    ref = oracle.combine_f64(oracle.bf16_bits_to_f64(yp), dr, w.astype(np.float64),
                             oracle.bf16_bits_to_f64(sh))
    # both are bf16 roundings of sums that differ by < k fp32 ulps: at most one
    # bf16 ulp apart
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-30))[1] - 8)
    assert np.all(np.abs(got - ref) <= ulp)
    assert np.mean(got == ref) > 0.95
    zero = np.zeros((T, k), np.float32)
    assert np.array_equal(oracle.combine_fma32(yp, dr, zero, sh), sh)


def test_combine_fma32_is_fused():
    # w*y = (1+2^-20)(1+2^-7) = 1 + 2^-7 + 2^-20 + 2^-27 needs 28 bits; with
    # acc = -(1+2^-7) a fused step keeps 2^-20 + 2^-27 (bf16-representable),
    # a rounded product followed by an add would give 2^-20.
    w = np.array([[1.0 + 2.0 ** -20]], np.float32)
    y = oracle.f64_to_bf16_bits(np.array([[1.0 + 2.0 ** -7]]))
    sh = oracle.f64_to_bf16_bits(np.array([[-(1.0 + 2.0 ** -7)]]))
    out = oracle.combine_fma32(y, np.array([0], np.int32), w, sh)
    assert oracle.bf16_bits_to_f64(out)[0, 0] == 2.0 ** -20 + 2.0 ** -27


# ------------------------------------------------------------------ expert FFN
def _ffn_closed_form_setup(g_vals, u_vals, H=16):
    """x = e_0 (one-hot); gate row i has g_vals[i] in column 0, up row i has
    u_vals[i] in column 0: G[:, i] = g_vals[i], U[:, i] = u_vals[i]."""
    I = len(g_vals)
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    wgu = np.zeros((2 * I, H))
    wgu[:I, 0] = g_vals
    wgu[I:, 0] = u_vals
    return x, wgu, I


def test_swiglu_closed_form_gate_and_up_roles():
    g = np.array([0.0, 2.0, -3.0, 0.5, 8.0, -0.25, 1.0, 4.0])
    u = np.array([3.0, 1.0, 1.0, -2.0, 0.5, 1.0, 0.0, -1.0])
    x, wgu, I = _ffn_closed_form_setup(g, u)
    wd = np.eye(16, I)                       # y[:, i] = h[:, i] for i < I
    h, y = oracle.swiglu_expert(x, wgu, wd, I)
    silu = torch.nn.functional.silu(torch.tensor(g, dtype=torch.float64)).numpy()
    want = oracle.bf16_round(silu * u)
    assert np.array_equal(h[0], want)
    assert h[0, 0] == 0.0                    # silu(0) = 0 whatever the up value
    assert h[0, 6] == 0.0                    # up = 0
    # swapping gate and up would give silu(u) * g; the data tell them apart
    assert not np.allclose(want, oracle.bf16_round(torch.nn.functional.silu(
        torch.tensor(u, dtype=torch.float64)).numpy() * g))
    assert np.array_equal(y[0, :I], h[0])
    assert np.all(y[0, I:] == 0)


def test_down_projection_orientation_with_permutation_matrix():
    rng = np.random.default_rng(9)
    H = I = 12
    x = oracle.bf16_round(rng.standard_normal((5, H)))
    wgu = oracle.bf16_round(rng.standard_normal((2 * I, H)) * 0.3)
    perm = rng.permutation(H)
    wd = np.zeros((H, I))
    wd[np.arange(H), perm] = 1.0             # output column c takes h[:, perm[c]]
    h, y = oracle.swiglu_expert(x, wgu, wd, I)
    assert np.array_equal(y, h[:, perm])


def test_grouped_ffn_uses_each_segments_expert():
    rng = np.random.default_rng(10)
    H = I = 8
    E = 3
    x = oracle.bf16_round(rng.standard_normal((10, H)))
    wgu_one = oracle.bf16_round(rng.standard_normal((2 * I, H)) * 0.5)
    wgu = np.stack([wgu_one] * E)
    wd = np.stack([(e + 1) * np.eye(H) for e in range(E)])
    offs = np.array([0, 3, 3, 10])           # an empty middle segment
    seg_expert = np.array([2, 0, 1])
    h, y = oracle.grouped_ffn(x, offs, seg_expert, wgu, wd, I)
    h1, _ = oracle.swiglu_expert(x, wgu_one, np.eye(H), I)
    assert np.array_equal(h, h1)
    np.testing.assert_array_equal(y[:3], oracle.bf16_round(3 * h1[:3]))
    np.testing.assert_array_equal(y[3:], oracle.bf16_round(2 * h1[3:]))
    # evaluating a subset of rows gives the same rows
    hs, ys = oracle.grouped_ffn(x, offs, seg_expert, wgu, wd, I, rows=np.array([1, 4, 9]))
    assert np.array_equal(ys, y[[1, 4, 9]])


def test_layer_on_sampled_tokens_matches_stagewise_oracle():
    """The per-token layer evaluation and the staged pipeline (route, layout,
    permute, grouped FFN, combine) agree: one reads the definition token by
    token, the other through the permutation."""
    w = wl.small_parity_workload(T=24, H=64, I=128, E=8, k=2, R=4)
    pl = wl.make_placement(w)
    lg = wl.make_logits(w).numpy()
    x = wl.make_x(w).view(torch.int16).numpy().view(np.uint16)
    wgu = wl.make_w_gate_up(w).view(torch.int16).numpy().view(np.uint16)
    wd = wl.make_w_down(w).view(torch.int16).numpy().view(np.uint16)
    ids, wts = oracle.route_softmax_topk(lg, w.k)
    lay = oracle.dispatch_layout(ids, pl)
    xp = oracle.bf16_bits_to_f64(oracle.permute(x, lay["dest_row"], w.k))
    _, yp = oracle.grouped_ffn(xp, lay["seg_offsets"], pl.slot_expert,
                               oracle.bf16_bits_to_f64(wgu), oracle.bf16_bits_to_f64(wd), w.I)
    y = oracle.combine_f64(yp, lay["dest_row"], wts.astype(np.float32).astype(np.float64))
    cfg = dict(score_fn=0, k=w.k, n_groups=1, topk_groups=1, group_topn=1)
    toks = [0, 5, 23]
    y2 = oracle.moe_layer_tokens(toks, lg, x, wgu, wd, pl, cfg, I=w.I)
    assert np.array_equal(y[toks], y2)


def test_balancedness_summed_across_layers():
    """"The slowest expert sets the pace": avg_tokens / max_tokens, summed
    across layers.  Two layers of the worked example's loads, the second
    mirrored: means 16 + 16, maxima 36 + 36, so 32/72 = 4/9 (summing the
    counts first would give 32/42 instead).  One layer reduces to the
    per-step statistic, identical layers to the one-layer value, and an
    empty step to 1.0."""
    a = np.array([36, 13, 9, 6])
    bal, mx, tot = oracle.balance_stats_layers(np.stack([a, a[::-1]]))
    assert (mx, tot) == (72, 128) and bal == 32.0 / 72.0
    assert bal != 32.0 / 42.0
    one = oracle.balance_stats_layers(a[None, :])
    assert one[0] == oracle.balance_stats(a)[0] == 16.0 / 36.0
    three = oracle.balance_stats_layers(np.stack([a, a, a]))
    assert three[0] == 16.0 / 36.0 and three[1:] == (108, 192)
    assert oracle.balance_stats_layers(np.zeros((3, 4), dtype=np.int32))[0] == 1.0
    assert oracle.balance_stats_layers(np.full((2, 8), 5))[0] == 1.0
