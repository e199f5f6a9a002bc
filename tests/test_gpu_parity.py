"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact: expert ids, slots, counts, offsets, permutation indices, rank
counts, balancedness, permuted rows, and the combine given the same expert
outputs (its fp32 fma order is fixed).  Floating outputs: relative
Frobenius error <= 1e-2 and, after normalising each row by its largest
|reference| value, max |err| <= 2e-2; router weights within 1e-6 relative
of fp64.
"""

import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

FROB_TOL = 1e-2
ROW_TOL = 2e-2
W_RTOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_ffn_gb300 import build
    build.build()
    oracle.build_c()
    torch.cuda.set_device(0)


def moe():
    from grouped_ffn_gb300 import moe as m
    return m


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits(t))


def assert_close(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / max(nrm, 1e-300)
    scale = np.max(np.abs(ref), axis=1)
    err = np.max(np.abs(got - ref), axis=1)
    row = np.where(scale > 0, err / np.where(scale > 0, scale, 1), err)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert rel <= FROB_TOL, f"{what}: rel Frobenius {rel:.3e}"
    assert row.max() <= ROW_TOL, f"{what}: per-row normalised max err {row.max():.3e} at row {row.argmax()}"
    return rel, row.max()


def bf16_ulps(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between two arrays of
    bf16-representable values (the GPU's bf16 output and the oracle's fp64
    result rounded to bf16): the difference of their positions on the
    ordered bf16 number line, on which -0 and +0 coincide."""
    def pos(v):
        b = oracle.f64_to_bf16_bits(np.asarray(v, np.float64)).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(pos(got) - pos(ref))


def assert_ulps(got: np.ndarray, ref: np.ndarray, what: str, within1: float, big_most: int):
    """The accuracy check on top of assert_close that would notice a loss of
    accuracy well inside it: at least a fraction `within1` of the elements
    within 1 bf16 ulp of the oracle, and no element whose reference is at
    least 1/64 of its row's largest magnitude more than `big_most` ulps away.
    Two correct roundings of the same sum in fp32 and in fp64 differ by at
    most one ulp, so a kernel that accumulates in fp32 and rounds once stays
    within 1 ulp except where the fp32 sum's own error crosses a rounding
    boundary.  Results that nearly cancel are the exception: there the fp32
    accumulator's error, tiny against the row's scale, can move the result by
    many of its own ulps or flip its sign, so the ulp bound is applied only
    away from zero."""
    got = np.asarray(got, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    u = bf16_ulps(got, ref)
    frac = float(np.mean(u <= 1)) if u.size else 1.0
    assert frac >= within1, f"{what}: only {frac:.5f} of elements within 1 bf16 ulp"
    big = np.abs(ref) >= np.abs(ref).max(axis=1, keepdims=True) / 64
    if big.any():
        worst = int(u[big].max())
        assert worst <= big_most, f"{what}: {worst} bf16 ulps away from zero"
    return frac


# Measured on GB300 against the oracle (sampled rows of the four full-size
# layers): h is within 1 ulp on 99.935-99.976% of elements and within 1 ulp
# wherever |h| >= max|h row| / 64; y_perm, one fp32 accumulation over h,
# within 1 ulp on 98.0-98.6% and at most 10 ulps away from zero.
H_WITHIN1, H_BIG_MOST = 0.999, 2
Y_WITHIN1, Y_BIG_MOST = 0.97, 16


def route_cfg(w):
    return moe().RouteCfg(w.score_fn, w.k, w.n_groups, w.topk_groups, w.group_topn)


def oracle_route(w, logits_np):
    if w.score_fn == wl.SCORE_SOFTMAX and w.n_groups == 1:
        ids, wts = oracle.route_softmax_topk(logits_np, w.k)
        return ids, wts, np.inf
    return oracle.route_group_limited(logits_np, w.k, w.n_groups, w.topk_groups, w.group_topn)


def gpu_route(w, logits):
    ids = torch.empty(w.T, w.k, dtype=torch.int32, device="cuda")
    wts = torch.empty(w.T, w.k, dtype=torch.float32, device="cuda")
    moe().moe_route(logits, route_cfg(w), ids, wts)
    return ids, wts


def gpu_layout(ids, pl_dev, T, k, ws=None):
    A = T * k
    m = moe()
    if ws is None:
        ws = m.new_workspace(T, k, pl_dev.n_slots)
    i32 = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
    out = dict(slot=i32(A), seg_counts=i32(pl_dev.n_slots), seg_offsets=i32(pl_dev.n_slots + 1),
               dest_row=i32(A), src_assign=i32(A), rank_counts=i32(pl_dev.n_ranks))
    m.moe_dispatch_layout(ids, pl_dev, out["slot"], out["seg_counts"], out["seg_offsets"],
                          out["dest_row"], out["src_assign"], out["rank_counts"], ws)
    m.moe_check_device_status(ws)
    return {k_: v.cpu().numpy() for k_, v in out.items()}


ALL = ["tiny", "decode", "prefill", "group_limited", "replica"]


# ------------------------------------------------------------------ route
@pytest.mark.parametrize("name,zipf", [(n, None) for n in ALL] +
                         [("replica", s) for s in (0.0, 0.5, 1.5)])
def test_route_parity(name, zipf):
    w = wl.WORKLOADS[name]
    if zipf is not None:
        w = w.with_zipf(zipf)
    logits = wl.make_logits(w, "cuda")
    ids, wts = gpu_route(w, logits)
    rid, rw, margin = oracle_route(w, logits.cpu().numpy())
    assert np.array_equal(ids.cpu().numpy(), rid), f"ids differ (min group margin {margin:.2e})"
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


@pytest.mark.parametrize("E,k,score", [(40, 16, 0), (33, 3, 0), (512, 16, 0), (64, 4, 1), (1, 1, 0), (16, 16, 1)])
def test_route_shapes_and_ties(E, k, score):
    rng = np.random.default_rng(E * 31 + k)
    T = 257
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 1.0], np.float32)
    lg = rng.choice(vals, size=(T, E)).astype(np.float32)     # many exact ties, signed zeros
    lg[: T // 2] = rng.standard_normal((T // 2, E)).astype(np.float32)
    w = wl.Workload("t", 0, T=T, H=8, E=E, k=k, I=8, R=1, ranks_per_node=1, score_fn=score)
    ids, wts = gpu_route(w, torch.from_numpy(lg).cuda())
    rid, rw, _ = oracle_route(w, lg)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


def test_route_group_limited_small_groups():
    rng = np.random.default_rng(3)
    for n_groups, E, topk_groups, topn, k in [(4, 64, 2, 3, 5), (32, 128, 3, 1, 4), (2, 40, 1, 2, 6)]:
        w = wl.Workload("g", 0, T=300, H=8, E=E, k=k, I=8, R=1, ranks_per_node=1,
                        score_fn=wl.SCORE_SIGMOID, n_groups=n_groups, topk_groups=topk_groups,
                        group_topn=topn)
        lg = rng.standard_normal((w.T, E)).astype(np.float32)
        ids, wts = gpu_route(w, torch.from_numpy(lg).cuda())
        rid, rw, _ = oracle_route(w, lg)
        assert np.array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


@pytest.mark.parametrize("n_groups,topk_groups,topn,k", [(16, 4, 2, 8), (8, 2, 1, 6), (32, 8, 3, 16),
                                                         (4, 4, 2, 8)])
def test_route_group_limited_full_width_other_group_shapes(n_groups, topk_groups, topn, k):
    """256 experts with other group shapes than the group-limited workload's
    (8 groups, top 4, sum of top 2), Zipf-skewed logits; the last case keeps
    every group, so it reduces to plain sigmoid top-k."""
    w = wl.WORKLOADS["group_limited"].scaled(T=2000, k=k, n_groups=n_groups,
                                             topk_groups=topk_groups, group_topn=topn)
    logits = wl.make_logits(w, "cuda")
    ids, wts = gpu_route(w, logits)
    rid, rw, _ = oracle_route(w, logits.cpu().numpy())
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


def test_route_group_limited_near_ties_decided_in_fp64():
    """Groups whose scores differ by less than fp32 can resolve: the kernel
    must fall back to the fp64 definition and agree with the oracle, and
    exact ties must go to the lower group id."""
    rng = np.random.default_rng(21)
    E, n_groups, gsz, T = 64, 8, 8, 512
    lg = np.full((T, E), -6.0, np.float32)
    one = np.float32(1.0)
    for t in range(T):
        a, b = rng.choice(n_groups, size=2, replace=False)
        ulps = int(rng.integers(0, 4))             # 0 = exact tie
        lg[t, a * gsz:a * gsz + 2] = [one, one]
        hi = one
        for _ in range(ulps):
            hi = np.nextafter(hi, np.float32(2.0))
        lg[t, b * gsz:b * gsz + 2] = [one, hi]
        lg[t, rng.integers(0, E)] += np.float32(rng.uniform(-1e-3, 0.0))   # noise elsewhere
    w = wl.Workload("nt", 0, T=T, H=8, E=E, k=2, I=8, R=1, ranks_per_node=1,
                    score_fn=wl.SCORE_SIGMOID, n_groups=n_groups, topk_groups=1, group_topn=2)
    ids, wts = gpu_route(w, torch.from_numpy(lg).cuda())
    rid, rw, margin = oracle_route(w, lg)
    assert margin < 1e-7                           # the cases really are near ties
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


@pytest.mark.parametrize("topn", [1, 2])
def test_route_groups_of_32_near_ties_and_repeated_maxima(topn):
    """Groups of exactly 32 experts (the group-limited layer's shape, whose
    group scores are merged across the warp in one pass): exact and
    one-to-three-ulp ties at the group cut must agree with the oracle
    (fp64 decides, ties to the lower group id), and a group whose largest
    logit appears twice scores it twice."""
    rng = np.random.default_rng(44 + topn)
    E, n_groups, gsz, T = 256, 8, 32, 1024
    lg = rng.normal(-4.0, 0.5, size=(T, E)).astype(np.float32)
    one = np.float32(1.0)
    for t in range(T):
        a, b, c = rng.choice(n_groups, size=3, replace=False)
        ulps = int(rng.integers(0, 4))             # 0 = exact tie
        hi = one
        for _ in range(ulps):
            hi = np.nextafter(hi, np.float32(2.0))
        la, lb = rng.choice(gsz, size=2, replace=False), rng.choice(gsz, size=2, replace=False)
        lg[t, a * gsz + la] = [one, one]
        lg[t, b * gsz + lb] = [one, hi] if topn == 2 else [hi, -9.0]
        lg[t, c * gsz + rng.choice(gsz, size=2, replace=False)] = [np.float32(3.0)] * 2
    w = wl.Workload("g32", 0, T=T, H=8, E=E, k=8, I=8, R=1, ranks_per_node=1,
                    score_fn=wl.SCORE_SIGMOID, n_groups=n_groups, topk_groups=2, group_topn=topn)
    ids, wts = gpu_route(w, torch.from_numpy(lg).cuda())
    rid, rw, margin = oracle_route(w, lg)
    assert margin < 1e-7                           # the cut really is a near tie
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=W_RTOL, atol=0)


# ------------------------------------------------------------------ layout + balance
@pytest.mark.parametrize("name,zipf", [(n, None) for n in ALL] +
                         [("replica", s) for s in (0.0, 0.5, 1.5)])
def test_layout_and_balance_parity(name, zipf):
    w = wl.WORKLOADS[name]
    if zipf is not None:
        w = w.with_zipf(zipf)
    pl = wl.make_placement(w)
    pl_dev = moe().DevicePlacement.from_tables(pl)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    ids_np = ids.cpu().numpy()
    got = gpu_layout(ids, pl_dev, w.T, w.k)
    ref = oracle.dispatch_layout(ids_np, pl)
    for key in ("slot", "seg_counts", "seg_offsets", "dest_row", "src_assign", "rank_counts"):
        assert np.array_equal(got[key], ref[key]), key
    b = torch.empty(1, dtype=torch.float64, device="cuda")
    mx = torch.empty(1, dtype=torch.int32, device="cuda")
    tot = torch.empty(1, dtype=torch.int64, device="cuda")
    moe().moe_balance_stats(torch.from_numpy(got["rank_counts"]).cuda(), b, mx, tot)
    assert (b.item(), mx.item(), tot.item()) == oracle.balance_stats(ref["rank_counts"])


def test_layout_many_tiles_many_slots_and_ragged_tail():
    # 100 tiles of 1024 assignments (the last one ragged), 1024 slots on 256 ranks
    T, k, E, R = 51111, 2, 1024, 256
    rng = np.random.default_rng(11)
    ids_np = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids_np[:, 1] = (ids_np[:, 0] + 1 + rng.integers(0, E - 1, size=T)) % E
    pl = wl.placement_from_hosts(E, R, 4, wl.round_robin_hosts(E, R))
    got = gpu_layout(torch.from_numpy(ids_np).cuda(), moe().DevicePlacement.from_tables(pl), T, k)
    ref = oracle.dispatch_layout(ids_np, pl)
    for key in ref:
        assert np.array_equal(got[key], ref[key]), key


def test_layout_tile_counts_in_turn_on_one_workspace():
    """276 tiles of 1024 assignments, then 8, 256, 3 and 257, then 276
    again, all on one workspace with no clearing in between: every call
    must leave the tile ticket and the look-back flags zero for the next
    one, whatever its tile count."""
    m = moe()
    E, R, k = 64, 8, 2
    pl = wl.placement_from_hosts(E, R, 8, wl.round_robin_hosts(E, R))
    pl_dev = m.DevicePlacement.from_tables(pl)
    rng = np.random.default_rng(33)
    T_max = 141_000                      # 282,000 assignments: 69 tiles
    ws = m.new_workspace(T_max, k, pl_dev.n_slots)
    for T in (T_max, 4001, 64 * 2048, 1500, 131_073, T_max):
        ids_np = rng.integers(0, E, size=(T, k)).astype(np.int32)
        ids_np[:, 1] = (ids_np[:, 0] + 1 + rng.integers(0, E - 1, size=T)) % E
        got = gpu_layout(torch.from_numpy(ids_np).cuda(), pl_dev, T, k, ws=ws)
        ref = oracle.dispatch_layout(ids_np, pl)
        for key in ref:
            assert np.array_equal(got[key], ref[key]), (T, key)


def test_layout_with_explicit_token_source_ranks():
    """The fixed replica rule with each token's rank given by an array
    instead of t mod R (tokens clustered on a few ranks, so that some nodes
    hold no copy of a hot expert and the spread rule applies)."""
    m = moe()
    w = wl.WORKLOADS["replica"].scaled(T=6000)
    base = wl.make_placement(w)
    rng = np.random.default_rng(21)
    src = rng.choice([0, 1, 5, 13], size=w.T).astype(np.int32)
    pl = wl.Placement(base.n_experts, base.n_ranks, base.ranks_per_node, base.slot_expert,
                      base.slot_rank, base.rep_offsets, base.rep_slots, src)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    got = gpu_layout(ids, m.DevicePlacement.from_tables(pl), w.T, w.k)
    ref = oracle.dispatch_layout(ids.cpu().numpy(), pl)
    for key in ("slot", "seg_counts", "seg_offsets", "dest_row", "src_assign", "rank_counts"):
        assert np.array_equal(got[key], ref[key]), key
    # the rule differs from t mod R here
    default = oracle.dispatch_layout(ids.cpu().numpy(), base)
    assert not np.array_equal(default["slot"], ref["slot"])


def test_layout_empty_and_single_token():
    pl = wl.make_placement(wl.WORKLOADS["tiny"])
    pl_dev = moe().DevicePlacement.from_tables(pl)
    got = gpu_layout(torch.empty(0, 2, dtype=torch.int32, device="cuda"), pl_dev, 0, 2)
    assert np.all(got["seg_counts"] == 0) and np.all(got["seg_offsets"] == 0)
    assert np.all(got["rank_counts"] == 0)
    one = np.array([[5, 63]], np.int32)
    got = gpu_layout(torch.from_numpy(one).cuda(), pl_dev, 1, 2)
    ref = oracle.dispatch_layout(one, pl)
    for key in ref:
        assert np.array_equal(got[key], ref[key]), key


def test_layout_is_deterministic_run_to_run():
    w = wl.WORKLOADS["replica"]
    pl_dev = moe().DevicePlacement.from_tables(wl.make_placement(w))
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    a = gpu_layout(ids, pl_dev, w.T, w.k)
    b = gpu_layout(ids, pl_dev, w.T, w.k)
    for key in a:
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("case", ["contiguous_pairs", "repack", "replicate_e0_on_rank3"])
def test_worked_example_on_gpu(case):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_example_balance.json")) as f:
        g = json.load(f)
    cs = g["cases"][case]
    ids_np = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(g["expert_counts"])])[:, None]
    T = ids_np.shape[0]
    if case == "replicate_e0_on_rank3":
        src = np.zeros(T, np.int32)
        src[np.nonzero(ids_np[:, 0] == 0)[0][1::2]] = 3
        pl = wl.placement_from_hosts(8, 4, 1, cs["hosts"], token_src_rank=src)
    else:
        pl = wl.placement_from_hosts(8, 4, 4, cs["hosts"])
    got = gpu_layout(torch.from_numpy(ids_np).cuda(), moe().DevicePlacement.from_tables(pl), T, 1)
    assert list(got["rank_counts"]) == cs["rank_loads"]
    b = torch.empty(1, dtype=torch.float64, device="cuda")
    mx = torch.empty(1, dtype=torch.int32, device="cuda")
    tot = torch.empty(1, dtype=torch.int64, device="cuda")
    moe().moe_balance_stats(torch.from_numpy(got["rank_counts"]).cuda(), b, mx, tot)
    assert b.item() == cs["balancedness_num"] / cs["balancedness_den"]


@pytest.mark.parametrize("L,R", [(1, 8), (2, 4), (7, 32), (61, 16), (3, 1024), (40, 1), (1, 1)])
def test_balance_stats_layers_bit_exact(L, R):
    """Balancedness summed across layers: the double, the sum of per-layer
    maxima and the total are the oracle's bit for bit; the mirrored worked
    example gives 4/9, one layer gives moe_balance_stats' value, and an
    empty step gives 1.0."""
    m = moe()
    rng = np.random.default_rng(L * 1000 + R)
    cases = [rng.integers(0, 5000, size=(L, R)).astype(np.int32),
             np.zeros((L, R), np.int32)]
    if (L, R) == (2, 4):
        cases.append(np.array([[36, 13, 9, 6], [6, 9, 13, 36]], np.int32))
    for rc in cases:
        b = torch.empty(1, dtype=torch.float64, device="cuda")
        mx = torch.empty(1, dtype=torch.int64, device="cuda")
        tot = torch.empty(1, dtype=torch.int64, device="cuda")
        m.moe_balance_stats_layers(torch.from_numpy(rc).cuda(), b, mx, tot)
        ref = oracle.balance_stats_layers(rc)
        assert (b.item(), int(mx.item()), int(tot.item())) == ref
        if rc.shape == (2, 4) and rc[0, 0] == 36:
            assert b.item() == 32.0 / 72.0
        if L == 1:
            b1 = torch.empty(1, dtype=torch.float64, device="cuda")
            mx1 = torch.empty(1, dtype=torch.int32, device="cuda")
            m.moe_balance_stats(torch.from_numpy(rc[0]).cuda(), b1, mx1, tot)
            assert b1.item() == b.item()


def test_layout_reports_bad_expert_id_without_faulting():
    m = moe()
    pl = wl.make_placement(wl.WORKLOADS["tiny"])
    pl_dev = m.DevicePlacement.from_tables(pl)
    ids = torch.tensor([[1, 2], [3, 64], [5, -1]], dtype=torch.int32, device="cuda")
    ws = m.new_workspace(3, 2, pl_dev.n_slots)
    A = 6
    o = [torch.zeros(n, dtype=torch.int32, device="cuda") for n in (A, 64, 65, A, A, 8)]
    m.moe_dispatch_layout(ids, pl_dev, *o, ws)
    with pytest.raises(m.MoeError) as ei:
        m.moe_check_device_status(ws)
    assert ei.value.status == 4
    m.moe_check_device_status(ws)   # cleared after reading


def test_bounded_waits_expire_report_and_leave_the_context_usable():
    """Failure detection without a fault: the grouped FFN's two kinds of
    bounded wait (an mbarrier phase, a global counter), run on conditions
    nothing satisfies, give up at their deadline, record
    MOE_ERR_DEVICE_TIMEOUT for the host, and leave the context usable."""
    m = moe()
    ws = m.new_workspace(8, 2, 64)
    waited = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    limit_us = 50_000
    t0 = time.perf_counter()
    m.moe_selftest_wait_timeout(ws, limit_us, waited)
    with pytest.raises(m.MoeError) as ei:
        m.moe_check_device_status(ws)
    wall = time.perf_counter() - t0
    assert ei.value.status == 5                          # MOE_ERR_DEVICE_TIMEOUT
    assert limit_us <= ei.value.info < limit_us + 500_000
    w = waited.cpu().tolist()
    assert all(limit_us <= x < limit_us + 500_000 for x in w), w
    assert wall < 10.0
    m.moe_check_device_status(ws)                        # reported once, then cleared
    # the same context still computes: permute then combine with one-hot
    # weights gives back the input bit for bit
    test_permute_then_combine_one_hot_is_identity()


# ------------------------------------------------------------------ permute / combine
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_permute_bit_exact(name):
    w = wl.WORKLOADS[name]
    m = moe()
    pl = wl.make_placement(w)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    lay = oracle.dispatch_layout(ids.cpu().numpy(), pl)
    x = wl.make_x(w, "cuda")
    xp = torch.empty(w.A, w.H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    m.moe_permute(x, w.k, torch.from_numpy(lay["dest_row"]).cuda(), xp, ws)
    m.moe_check_device_status(ws)
    assert np.array_equal(bits(xp), oracle.permute(bits(x), lay["dest_row"], w.k))


@pytest.mark.parametrize("k,H,shared", [(2, 256, False), (4, 4096, False), (8, 7168, True),
                                        (3, 136, True), (16, 64, False), (1, 520, True),
                                        (1, 8192, False)])
def test_combine_bit_exact(k, H, shared):
    m = moe()
    T = 333
    g = torch.Generator(device="cuda").manual_seed(k * 1000 + H)
    yp = torch.randn(T * k, H, generator=g, device="cuda").to(torch.bfloat16)
    sh = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16) if shared else None
    dr = torch.randperm(T * k, generator=g, device="cuda").to(torch.int32)
    wts = torch.rand(T, k, generator=g, device="cuda")
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(T, k, 1)
    m.moe_combine(yp, dr, wts, y, ws, sh)
    m.moe_check_device_status(ws)
    ref = oracle.combine_fma32(bits(yp), dr.cpu().numpy(), wts.cpu().numpy(),
                               None if sh is None else bits(sh))
    assert np.array_equal(bits(y), ref)


@pytest.mark.parametrize("T,H,k", [(37, 136, 3), (5, 8, 1), (300, 4104, 2)])
def test_permute_odd_widths_bit_exact(T, H, k):
    """Row widths that are not a multiple of the copy loop's unroll (H/8 =
    17, 1 and 513 chunks of 16 bytes)."""
    m = moe()
    g = torch.Generator(device="cuda").manual_seed(T + H)
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    dr = torch.randperm(T * k, generator=g, device="cuda").to(torch.int32)
    xp = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(T, k, 1)
    m.moe_permute(x, k, dr, xp, ws)
    m.moe_check_device_status(ws)
    assert np.array_equal(bits(xp), oracle.permute(bits(x), dr.cpu().numpy(), k))


def test_permute_then_combine_one_hot_is_identity():
    m = moe()
    w = wl.WORKLOADS["replica"]
    pl = wl.make_placement(w)
    pl_dev = m.DevicePlacement.from_tables(pl)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    dest = torch.empty(w.A, dtype=torch.int32, device="cuda")
    scratch = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (w.A, pl.n_slots, pl.n_slots + 1)]
    src = torch.empty(w.A, dtype=torch.int32, device="cuda")
    rc = torch.empty(w.R, dtype=torch.int32, device="cuda")
    m.moe_dispatch_layout(ids, pl_dev, scratch[0], scratch[1], scratch[2], dest, src, rc, ws)
    x = wl.make_x(w, "cuda")
    xp = torch.empty(w.A, w.H, dtype=torch.bfloat16, device="cuda")
    m.moe_permute(x, w.k, dest, xp, ws)
    onehot = torch.zeros(w.T, w.k, device="cuda")
    onehot[:, w.k - 1] = 1.0
    y = torch.empty_like(x)
    m.moe_combine(xp, dest, onehot, y, ws)
    m.moe_check_device_status(ws)
    assert torch.equal(y, x)


# ------------------------------------------------------------------ grouped FFN
def _ffn_case(w, offsets, seg_expert, dev="cuda"):
    m = moe()
    n_rows = int(offsets[-1]) + 37          # rows past the last segment stay unwritten
    g = torch.Generator(device=dev).manual_seed(w.index)
    xp = torch.randn(n_rows, w.H, generator=g, device=dev).to(torch.bfloat16)
    wgu = wl.make_w_gate_up(w, dev)
    wd = wl.make_w_down(w, dev)
    h = torch.full((n_rows, w.I), float("nan"), dtype=torch.bfloat16, device=dev)
    yp = torch.full((n_rows, w.H), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = m.new_workspace(1, 1, len(seg_expert))
    offs_t = torch.tensor(offsets, dtype=torch.int32, device=dev)
    exp_t = torch.tensor(seg_expert, dtype=torch.int32, device=dev)
    m.moe_grouped_ffn(xp, offs_t, exp_t, wgu, wd, h, yp, ws)
    m.moe_check_device_status(ws)
    rh, ry = oracle.grouped_ffn(f64(xp[: offsets[-1]]), np.array(offsets), np.array(seg_expert),
                                oracle.bf16_bits_to_f64(bits(wgu)), oracle.bf16_bits_to_f64(bits(wd)),
                                w.I)
    return h, yp, rh, ry, n_rows


@pytest.mark.parametrize("H,I,counts", [
    (256, 128, [3, 0, 5, 8]),                          # tiny layer shape, fewer rows than a tile
    (512, 384, [130, 1, 0, 257, 128, 75, 300, 12]),    # several tiles, ragged tails, empty
    (768, 256, [600]),                                 # one segment = a dense GEMM
    (256, 640, [129, 127, 2, 64]),
])
def test_grouped_ffn_small_full_compare(H, I, counts):
    E = len(counts) + 1
    w = wl.Workload("ffn", 50 + H // 256 + I, T=1, H=H, E=E, k=1, I=I, R=1, ranks_per_node=1)
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    seg_expert = [(3 * s + 1) % E for s in range(len(counts))]
    h, yp, rh, ry, n_rows = _ffn_case(w, offsets, seg_expert)
    A = offsets[-1]
    assert_close(f64(h[:A]), rh, "h")
    assert_close(f64(yp[:A]), ry, "y_perm")
    assert_ulps(f64(h[:A]), rh, "h", H_WITHIN1, H_BIG_MOST)
    assert_ulps(f64(yp[:A]), ry, "y_perm", Y_WITHIN1, Y_BIG_MOST)
    assert torch.isnan(yp[A:].float()).all() and torch.isnan(h[A:].float()).all()


def test_grouped_ffn_at_the_segment_limit():
    """1024 segments (the limit), most empty or one row, a few long and
    ragged, mapped onto 33 experts (segments may share an expert): the
    device-side tile list over all of them, compared in full."""
    m = moe()
    S, E, H, I = 1024, 33, 256, 128
    rng = np.random.default_rng(11)
    counts = rng.choice([0, 0, 0, 1, 1, 2, 5], size=S)
    counts[[3, 500, 1023]] = [300, 129, 257]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    seg_expert = ((np.arange(S) * 7) % E).astype(np.int32)
    w = wl.Workload("segmax", 61, T=1, H=H, E=E, k=1, I=I, R=1, ranks_per_node=1)
    A = int(offsets[-1])
    g = torch.Generator(device="cuda").manual_seed(61)
    xp = torch.randn(A, H, generator=g, device="cuda").to(torch.bfloat16)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    h = torch.empty(A, I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(A, H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, S)
    m.moe_grouped_ffn_packed(xp, torch.from_numpy(offsets).cuda(), torch.from_numpy(seg_expert).cuda(),
                             pgu, pd, h, y, ws)
    m.moe_check_device_status(ws)
    rh, ry = oracle.grouped_ffn(f64(xp), offsets, seg_expert, oracle.bf16_bits_to_f64(bits(wgu)),
                                oracle.bf16_bits_to_f64(bits(wd)), I)
    assert_close(f64(h), rh, "h (1024 segments)")
    assert_close(f64(y), ry, "y_perm (1024 segments)")
    assert_ulps(f64(h), rh, "h (1024 segments)", H_WITHIN1, H_BIG_MOST)
    assert_ulps(f64(y), ry, "y_perm (1024 segments)", Y_WITHIN1, Y_BIG_MOST)


def test_grouped_ffn_with_no_rows_launches_nothing():
    m = moe()
    w = wl.Workload("ffn0", 62, T=1, H=256, E=2, k=1, I=128, R=1, ranks_per_node=1)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    h = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    xp = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, 2)
    offs = torch.zeros(3, dtype=torch.int32, device="cuda")
    m.moe_grouped_ffn(xp, offs, torch.zeros(2, dtype=torch.int32, device="cuda"), wgu, wd, h, y, ws)
    m.moe_check_device_status(ws)


def test_grouped_ffn_reports_a_bad_expert_and_computes_the_rest():
    """A non-empty segment whose expert id is out of range is reported
    (MOE_ERR_DEVICE_INDEX) and skipped, without a fault; the other segments'
    rows are still right."""
    m = moe()
    H, I, E = 256, 128, 3
    counts = [40, 25, 130]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    A = int(offsets[-1])
    w = wl.Workload("ffnbad", 63, T=1, H=H, E=E, k=1, I=I, R=1, ranks_per_node=1)
    g = torch.Generator(device="cuda").manual_seed(63)
    xp = torch.randn(A, H, generator=g, device="cuda").to(torch.bfloat16)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    h = torch.full((A, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((A, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    seg_expert = np.array([2, 7, 0], np.int32)          # segment 1 names expert 7 of 3
    ws = m.new_workspace(1, 1, 3)
    m.moe_grouped_ffn(xp, torch.from_numpy(offsets).cuda(), torch.from_numpy(seg_expert).cuda(),
                      wgu, wd, h, y, ws)
    with pytest.raises(m.MoeError) as ei:
        m.moe_check_device_status(ws)
    assert ei.value.status == 4
    good = np.r_[0:40, 65:195]
    ok_exp = np.array([2, 0, 0], np.int32)             # any valid id for the skipped segment
    rh, ry = oracle.grouped_ffn(f64(xp), offsets, ok_exp, oracle.bf16_bits_to_f64(bits(wgu)),
                                oracle.bf16_bits_to_f64(bits(wd)), I)
    gt = torch.from_numpy(good).cuda()
    assert_close(f64(y[gt]), ry[good], "y_perm of the valid segments")
    assert torch.isnan(y[40:65].float()).all()         # the bad segment is left unwritten


@pytest.mark.parametrize("H,I,counts", [(256, 128, [3, 0, 5, 8]),
                                         (512, 384, [130, 1, 0, 257, 128, 75, 300, 12])])
def test_packed_ffn_is_bit_identical_to_plain(H, I, counts):
    m = moe()
    E = len(counts) + 1
    w = wl.Workload("ffnp", 70 + H // 256 + I, T=1, H=H, E=E, k=1, I=I, R=1, ranks_per_node=1)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    se = torch.tensor([(5 * s + 2) % E for s in range(len(counts))], dtype=torch.int32, device="cuda")
    n = int(offs[-1]) + 5
    g = torch.Generator(device="cuda").manual_seed(3)
    xp = torch.randn(n, H, generator=g, device="cuda").to(torch.bfloat16)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    # the packed layout, as the header defines it
    NB1, nk1, NB2, nk2 = I // 128, H // 64, H // 256, I // 64
    want_gu = wgu.view(E, 2, NB1, 128, nk1, 64).permute(0, 2, 4, 1, 3, 5).reshape(E, 2 * I, H)
    want_d = wd.view(E, NB2, 2, 128, nk2, 64).permute(0, 1, 4, 2, 3, 5).reshape(E, H, I)
    assert torch.equal(pgu, want_gu) and torch.equal(pd, want_d)
    ws = m.new_workspace(1, 1, len(counts))
    outs = []
    for fn, a, b in ((m.moe_grouped_ffn, wgu, wd), (m.moe_grouped_ffn_packed, pgu, pd)):
        h = torch.zeros(n, I, dtype=torch.bfloat16, device="cuda")
        y = torch.zeros(n, H, dtype=torch.bfloat16, device="cuda")
        fn(xp, offs, se, a, b, h, y, ws)
        outs.append((h, y))
    m.moe_check_device_status(ws)
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def _sample_rows(seg_offsets, rng, n=48):
    A = int(seg_offsets[-1])
    rows = set(rng.choice(A, size=min(n, A), replace=False).tolist())
    for s in range(len(seg_offsets) - 1):      # first and last row of some segments
        lo, hi = int(seg_offsets[s]), int(seg_offsets[s + 1])
        if hi > lo and len(rows) < 2 * n:
            rows.update([lo, hi - 1])
    return np.array(sorted(rows))


class _LazyExperts:
    """Copies one expert's weights to the host on first use."""

    def __init__(self, t):
        self.t, self.cache = t, {}

    def __getitem__(self, e):
        if e not in self.cache:
            self.cache[e] = oracle.bf16_bits_to_f64(bits(self.t[e]))
        return self.cache[e]


def _full_layer(w, dev="cuda"):
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    pl = wl.make_placement(w)
    logits = wl.make_logits(w, dev)
    x = wl.make_x(w, dev)
    wgu = wl.make_w_gate_up(w, dev)
    wd = wl.make_w_down(w, dev)
    sgu, sd = wl.make_shared_weights(w, dev)
    layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl, dev),
                     w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                     n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                     shared_w_gate_up=sgu, shared_w_down=sd, device=dev)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
    layer.forward(logits, x, y)
    layer.check()
    torch.cuda.synchronize()
    return pl, logits, x, wgu, wd, sgu, sd, layer, y


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "group_limited", "replica"])
def test_full_layer_sampled(name):
    """Full-size layer in the configuration the benchmark times: every
    integer output bit-exact, FFN rows and combined tokens against the
    oracle (all of them on tiny and decode, sampled on the larger layers),
    and the combine bit-exact given the GPU's expert outputs."""
    w = wl.WORKLOADS[name]
    pl, logits, x, wgu, wd, sgu, sd, layer, y = _full_layer(w)
    A = w.A
    ids_ref, _, _ = oracle_route(w, logits.cpu().numpy())
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    lay = oracle.dispatch_layout(ids_ref, pl)
    for key in ("seg_counts", "seg_offsets", "rank_counts"):
        assert np.array_equal(getattr(layer, key).cpu().numpy(), lay[key]), key
    assert np.array_equal(layer.dest_row[:A].cpu().numpy(), lay["dest_row"])
    assert np.array_equal(layer.src_assign[:A].cpu().numpy(), lay["src_assign"])
    rng = np.random.default_rng(w.index)
    # rows of the grouped FFN (x_perm -> h, y_perm): all of them on the small
    # layers (tiny, decode), sampled on the large ones
    rows = np.arange(A) if A <= 256 else _sample_rows(lay["seg_offsets"], rng)
    xp_rows = f64(layer.x_perm[torch.from_numpy(rows).cuda()])
    lazy_gu, lazy_d = _LazyExperts(wgu), _LazyExperts(wd)
    full_x = np.zeros((int(rows.max()) + 1, w.H))
    full_x[rows] = xp_rows
    rh, ry = oracle.grouped_ffn(full_x, lay["seg_offsets"], pl.slot_expert, lazy_gu, lazy_d, w.I,
                                rows=rows)
    assert_close(f64(layer.h[torch.from_numpy(rows).cuda()]), rh, "h rows")
    assert_close(f64(layer.y_perm[torch.from_numpy(rows).cuda()]), ry, "y_perm rows")
    assert_ulps(f64(layer.h[torch.from_numpy(rows).cuda()]), rh, "h rows", H_WITHIN1, H_BIG_MOST)
    assert_ulps(f64(layer.y_perm[torch.from_numpy(rows).cuda()]), ry, "y_perm rows", Y_WITHIN1, Y_BIG_MOST)
    # combine bit-exact from the GPU's own expert outputs
    shared_out = layer.shared_output(w.T)
    shared_bits = bits(shared_out) if shared_out is not None else None
    ref_y = oracle.combine_fma32(bits(layer.y_perm[:A]), lay["dest_row"],
                                 layer.topk_w[: w.T].cpu().numpy(), shared_bits)
    assert np.array_equal(bits(y), ref_y)
    # whole layer on sampled tokens, from the definition
    toks = (np.arange(w.T) if w.T <= 64 else
            np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, size=12, replace=False)])))
    cfg = dict(score_fn=w.score_fn, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
               group_topn=w.group_topn)
    shared = None if sgu is None else (bits(sgu[0]), bits(sd[0]))
    ref = oracle.moe_layer_tokens(toks, logits.cpu().numpy(), bits(x), _BitsExperts(wgu),
                                  _BitsExperts(wd), pl, cfg, shared_w=shared, I=w.I,
                                  shared_I=w.shared_I)
    assert_close(f64(y[torch.from_numpy(toks).cuda()]), ref, "layer output")
    bal, mx, tot = oracle.balance_stats(lay["rank_counts"])
    assert layer.balancedness.item() == bal and layer.max_count.item() == mx
    assert layer.total.item() == tot == A


def _random_workload(seed: int) -> wl.Workload:
    """A seeded random small layer: hidden, intermediate, expert count, top-k,
    tokens, ranks and skew vary; every third is group-limited (sigmoid), and
    every fourth has a shared expert of the routed width (run in the routed
    launch)."""
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.choice([256, 512, 768, 1024]))
    I = int(rng.choice([128, 256, 384, 512]))
    if seed % 3 == 2:
        n_groups = int(rng.choice([2, 4, 8]))
        per = int(rng.choice([4, 8, 16]))
        E = n_groups * per
        topk_groups = int(rng.integers(1, n_groups + 1))
        group_topn = int(rng.integers(1, min(3, per) + 1))
        k = int(rng.integers(1, min(8, topk_groups * per) + 1))
        score = wl.SCORE_SIGMOID
    else:
        E = int(rng.integers(1, 81))
        k = int(rng.integers(1, min(8, E) + 1))
        n_groups = topk_groups = group_topn = 1
        score = wl.SCORE_SOFTMAX
    R = int(rng.choice([1, 2, 4, 8]))
    return wl.Workload(f"random{seed}", 100 + seed, T=int(rng.integers(1, 301)), H=H, E=E, k=k, I=I,
                       R=R, ranks_per_node=R, score_fn=score, n_groups=n_groups,
                       topk_groups=topk_groups, group_topn=group_topn,
                       shared_I=I if seed % 4 == 1 else 0,
                       zipf_s=float(rng.choice([0.0, 0.5, 1.0, 1.5])))


@pytest.mark.parametrize("seed", range(32))
def test_random_small_layers_against_the_oracle(seed):
    """Seeded random small layers: every integer output bit-exact and every
    token's output within tolerance of the oracle's token-by-token
    definition.  Such layers have fewer FFN tiles than CTAs or a ragged last
    wave, one-tile layouts, k = 1, single experts and empty experts."""
    w = _random_workload(seed)
    pl, logits, x, wgu, wd, sgu, sd, layer, y = _full_layer(w)
    A = w.A
    ids_ref, _, _ = oracle_route(w, logits.cpu().numpy())
    assert np.array_equal(layer.topk_ids[: w.T].cpu().numpy(), ids_ref), w
    lay = oracle.dispatch_layout(ids_ref, pl)
    for key in ("seg_counts", "seg_offsets", "rank_counts"):
        assert np.array_equal(getattr(layer, key).cpu().numpy(), lay[key]), (key, w)
    assert np.array_equal(layer.dest_row[:A].cpu().numpy(), lay["dest_row"])
    assert np.array_equal(layer.src_assign[:A].cpu().numpy(), lay["src_assign"])
    cfg = dict(score_fn=w.score_fn, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
               group_topn=w.group_topn)
    shared = None if sgu is None else (bits(sgu[0]), bits(sd[0]))
    ref = oracle.moe_layer_tokens(np.arange(w.T), logits.cpu().numpy(), bits(x), _BitsExperts(wgu),
                                  _BitsExperts(wd), pl, cfg, shared_w=shared, I=w.I,
                                  shared_I=w.shared_I)
    assert_close(f64(y), ref, f"layer output of {w}")
    bal, mx, tot = oracle.balance_stats(lay["rank_counts"])
    assert layer.balancedness.item() == bal and layer.max_count.item() == mx
    assert layer.total.item() == tot == A


@pytest.mark.parametrize("seed", range(12))
def test_random_small_layers_variants_are_bit_identical(seed):
    """On the same random layers, every variant path gives the plain step's
    output bits: rows gathered straight from x (no permute), the
    fixed-capacity layout with a capacity no slot exceeds (no drops), plain
    (unpacked) weights, the shared expert as a second launch, and the step
    replayed as one CUDA graph."""
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = _random_workload(seed)
    pl = wl.make_placement(w)
    dp = m.DevicePlacement.from_tables(pl)
    logits, x = wl.make_logits(w, "cuda"), wl.make_x(w, "cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    sgu, sd = wl.make_shared_weights(w, "cuda")

    def run(**kw):
        layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=dp, w_gate_up=wgu, w_down=wd,
                         max_tokens=w.T, score_fn=w.score_fn, n_groups=w.n_groups,
                         topk_groups=w.topk_groups, group_topn=w.group_topn,
                         shared_w_gate_up=sgu, shared_w_down=sd, **kw)
        y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        layer.forward(logits, x, y)
        layer.check()
        return layer, y

    base_layer, base = run()
    cap = max(1, int(base_layer.seg_counts.max().item()))
    variants = {"unpacked": dict(packed=False), "two launches": dict(fuse_shared=False),
                "gather": dict(gather=True), "fixed capacity %d" % cap: dict(masked_cap=cap)}
    for name, kw in variants.items():
        _, y = run(**kw)
        assert torch.equal(y, base), (name, w)
    graph = base_layer.capture(logits, x, base)
    out = base.clone()
    base.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(base, out), ("graph replay", w)


class _BitsExperts:
    """Copies one expert's bf16 bits to the host on first use."""

    def __init__(self, t):
        self.t, self.cache = t, {}

    def __getitem__(self, e):
        if e not in self.cache:
            self.cache[e] = bits(self.t[e])
        return self.cache[e]


def test_shared_expert_in_the_routed_launch():
    """moe_permute_shared copies every token once more after the dispatched
    rows, and moe_grouped_ffn_packed_shared runs the shared expert on those
    rows in the routed experts' launch: the copied rows are bit-exact, the
    shared rows match the dense definition, and the routed rows are the
    bits of a launch without the extra segment."""
    m = moe()
    T, k, H, I, E = 300, 2, 512, 256, 5
    w = wl.Workload("shfused", 64, T=T, H=H, E=E + 1, k=k, I=I, R=1, ranks_per_node=1)
    A = T * k
    g = torch.Generator(device="cuda").manual_seed(64)
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    dest = torch.randperm(A, generator=g, device="cuda").to(torch.int32)
    counts = [130, 0, 257, 1, 212]
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    se = torch.tensor([4, 0, 2, 1, 3], dtype=torch.int32, device="cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")   # expert E is the shared one
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    ws = m.new_workspace(T, k, len(counts) + 1)
    xp = torch.empty(A + T, H, dtype=torch.bfloat16, device="cuda")
    m.moe_permute_shared(x, k, dest, xp, ws)
    m.moe_check_device_status(ws)
    xb = bits(x)
    assert np.array_equal(bits(xp[:A]), oracle.permute(xb, dest.cpu().numpy(), k))
    assert np.array_equal(bits(xp[A:]), xb)
    h = torch.empty(A + T, I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(A + T, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_ffn_packed_shared(xp, offs, se, pgu, pd, A, T, E, h, y, ws)
    m.moe_check_device_status(ws)
    _, ry = oracle.swiglu_expert(f64(x), f64(wgu[E]), f64(wd[E]), I)
    assert_close(f64(y[A:]), ry, "shared expert rows")
    h2 = torch.empty(A, I, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(A, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_ffn_packed(xp[:A].contiguous(), offs, se, pgu, pd, h2, y2, ws)
    m.moe_check_device_status(ws)
    assert torch.equal(h[:A], h2) and torch.equal(y[:A], y2)


def test_fused_shared_layer_is_bit_identical_to_two_launches():
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = wl.WORKLOADS["group_limited"].scaled(T=512, E=64, R=16, H=1024, I=256, shared_I=256)
    pl = wl.make_placement(w)
    logits, x = wl.make_logits(w, "cuda"), wl.make_x(w, "cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    sgu, sd = wl.make_shared_weights(w, "cuda")
    outs = []
    for fuse in (True, False):
        layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl),
                         w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                         n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                         shared_w_gate_up=sgu, shared_w_down=sd, fuse_shared=fuse)
        assert layer.fuse_shared == fuse
        y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        layer.forward(logits, x, y)
        layer.check()
        outs.append((y, layer.shared_output(w.T).clone(), layer.launches_per_step))
        del layer
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert outs[0][2] == outs[1][2] - 1


def test_shared_expert_alone_matches_dense_definition():
    """The shared expert is one segment covering every token."""
    w = wl.WORKLOADS["group_limited"].scaled(T=200, H=512, I=256, shared_I=256, E=8)
    m = moe()
    x = wl.make_x(w, "cuda")
    sgu, sd = wl.make_shared_weights(w, "cuda")
    h = torch.empty(w.T, w.shared_I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, 1)
    m.moe_grouped_ffn(x, torch.tensor([0, w.T], dtype=torch.int32, device="cuda"),
                      torch.zeros(1, dtype=torch.int32, device="cuda"), sgu, sd, h, y, ws)
    m.moe_check_device_status(ws)
    rh, ry = oracle.swiglu_expert(f64(x), f64(sgu[0]), f64(sd[0]), w.shared_I)
    assert_close(f64(y), ry, "shared y")


# ------------------------------------------------------------------ replica routing (water-filling)
def _gpu_route_replicas(ids, pl, c):
    m = moe()
    pl_dev = m.DevicePlacement.from_tables(pl)
    T, k = ids.shape
    ws = m.new_workspace(T, k, pl.n_slots, n_experts=pl.n_experts, n_ranks=pl.n_ranks)
    slot = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    inter = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    m.moe_route_replicas(ids, pl_dev, c[0], c[1], slot, inter, ws)
    m.moe_check_device_status(ws)
    return slot, int(inter.item()), pl_dev, ws


@pytest.mark.parametrize("zipf,c", [(1.0, (0, 1)), (1.0, (1, 10)), (1.0, (1, 1)), (0.0, (1, 4)),
                                    (1.5, (3, 10))])
def test_route_replicas_parity(zipf, c):
    w = wl.WORKLOADS["replica"].with_zipf(zipf)
    pl = wl.make_placement(w)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    ids_np = ids.cpu().numpy()
    slot, inter, pl_dev, ws = _gpu_route_replicas(ids, pl, c)
    ref_slot, ref_inter = oracle.route_replicas_waterfill(ids_np, pl, *c)
    assert np.array_equal(slot.cpu().numpy(), ref_slot)
    assert inter == ref_inter
    # the layout from these slots, on the same workspace
    m = moe()
    A, S, R = w.A, pl.n_slots, w.R
    out = [torch.full((n,), -7, dtype=torch.int32, device="cuda") for n in (S, S + 1, A, A, R)]
    m.moe_dispatch_layout_routed(ids, slot, pl_dev, *out, ws)
    m.moe_check_device_status(ws)
    ref = oracle.dispatch_layout_from_slots(ids_np, ref_slot, pl)
    for key, t in zip(("seg_counts", "seg_offsets", "dest_row", "src_assign", "rank_counts"), out):
        assert np.array_equal(t.cpu().numpy(), ref[key]), key


def test_route_replicas_skewed_sources_and_figure6():
    rng = np.random.default_rng(5)
    # tokens concentrated on node 0: local replicas overflow their bounds
    w = wl.WORKLOADS["replica"].scaled(T=3000)
    hosts = wl.replica_hosts(w)
    src = np.where(rng.random(w.T) < 0.7, rng.integers(0, 4, w.T), rng.integers(0, 16, w.T))
    pl = wl.placement_from_hosts(w.E, w.R, w.ranks_per_node, hosts, token_src_rank=src)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    for c in [(0, 1), (1, 5), (2, 1)]:
        slot, inter, _, _ = _gpu_route_replicas(ids, pl, c)
        ref_slot, ref_inter = oracle.route_replicas_waterfill(ids.cpu().numpy(), pl, *c)
        assert np.array_equal(slot.cpu().numpy(), ref_slot) and inter == ref_inter
    # the "Zepp" Figure 6 scenario
    R, rpn = 8, 2
    src = np.concatenate([np.arange(16) % R] * 2)
    pl = wl.placement_from_hosts(2, R, rpn, [[0, 2, 4, 6], [1, 3, 5]], token_src_rank=src)
    ids6 = torch.tensor(np.concatenate([np.zeros(16), np.ones(16)]).astype(np.int32)[:, None],
                        device="cuda")
    slot, inter, _, _ = _gpu_route_replicas(ids6, pl, (1, 1))
    ref_slot, ref_inter = oracle.route_replicas_waterfill(ids6.cpu().numpy(), pl, 1, 1)
    assert np.array_equal(slot.cpu().numpy(), ref_slot) and inter == ref_inter == 4


def _gpu_refine(ids, pl_dev, slot, ws):
    m = moe()
    msgs = torch.full((2,), -9, dtype=torch.int32, device="cuda")
    m.moe_route_refine(ids, pl_dev, slot, msgs, ws)
    m.moe_check_device_status(ws)
    return slot, tuple(int(v) for v in msgs.cpu())


@pytest.mark.parametrize("zipf", [0.0, 0.5, 1.0, 1.5])
def test_route_refine_parity_replica_workload(zipf):
    """The consolidation refinement ("Zepp", Section 5) on the full replica
    workload at each exponent of the sweep: slots and message counts
    bit-exact against the oracle, per-copy loads unchanged, and the layout
    from the refined slots on the same workspace."""
    w = wl.WORKLOADS["replica"].with_zipf(zipf)
    pl = wl.make_placement(w)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    ids_np = ids.cpu().numpy()
    slot, inter, pl_dev, ws = _gpu_route_replicas(ids, pl, (1, 10))
    ref_in, ref_inter = oracle.route_replicas_waterfill(ids_np, pl, 1, 10)
    ref_slot, before, after = oracle.refine_consolidate(ids_np, ref_in, pl)
    slot, msgs = _gpu_refine(ids, pl_dev, slot, ws)
    assert np.array_equal(slot.cpu().numpy(), ref_slot)
    assert msgs == (before, after) and after < before
    assert np.array_equal(np.bincount(ref_slot, minlength=pl.n_slots),
                          np.bincount(ref_in, minlength=pl.n_slots))
    m = moe()
    A, S, R = w.A, pl.n_slots, w.R
    out = [torch.full((n,), -7, dtype=torch.int32, device="cuda") for n in (S, S + 1, A, A, R)]
    m.moe_dispatch_layout_routed(ids, slot, pl_dev, *out, ws)
    m.moe_check_device_status(ws)
    ref = oracle.dispatch_layout_from_slots(ids_np, ref_slot, pl)
    for key, t in zip(("seg_counts", "seg_offsets", "dest_row", "src_assign", "rank_counts"), out):
        assert np.array_equal(t.cpu().numpy(), ref[key]), key


def test_route_refine_hand_worked_and_explicit_sources():
    """The hand-worked refinement cases of the oracle's pins, and a
    replica-shaped layer with skewed explicit source ranks, on the GPU."""
    cases = [([[1, 2], [2, 3], [0]], [[0, 1], [0, 2], [2, 1]], [2, 2, 1, 0, 0, 3], (4, 3)),
             ([[1, 2], [1, 2], [0]], [[0, 1], [0, 2], [2, 1]], [1, 1, 2, 0, 0, 2], (3, 3)),
             ([[1, 3], [0], [0], [3]], [[3, 0], [0, 2]], [3, 3, 1, 0], (3, 2))]
    for hosts, ids_l, want_ranks, want_msgs in cases:
        ids_np = np.array(ids_l, dtype=np.int32)
        src = np.zeros(ids_np.shape[0], dtype=np.int32)
        pl = wl.placement_from_hosts(len(hosts), 4, 1, hosts, token_src_rank=src)
        ids = torch.tensor(ids_np, device="cuda")
        slot, _, pl_dev, ws = _gpu_route_replicas(ids, pl, (0, 1))
        slot, msgs = _gpu_refine(ids, pl_dev, slot, ws)
        assert [int(pl.slot_rank[s]) for s in slot.cpu().numpy()] == want_ranks
        assert msgs == want_msgs
    rng = np.random.default_rng(11)
    w = wl.WORKLOADS["replica"].scaled(T=5000)
    hosts = wl.replica_hosts(w)
    src = np.where(rng.random(w.T) < 0.6, rng.integers(0, 4, w.T), rng.integers(0, 16, w.T))
    pl = wl.placement_from_hosts(w.E, w.R, w.ranks_per_node, hosts, token_src_rank=src)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    for c in [(0, 1), (1, 5)]:
        slot, _, pl_dev, ws = _gpu_route_replicas(ids, pl, c)
        ref_in, _ = oracle.route_replicas_waterfill(ids.cpu().numpy(), pl, *c)
        ref_slot, before, after = oracle.refine_consolidate(ids.cpu().numpy(), ref_in, pl)
        slot, msgs = _gpu_refine(ids, pl_dev, slot, ws)
        assert np.array_equal(slot.cpu().numpy(), ref_slot) and msgs == (before, after)


@pytest.mark.parametrize("seed", list(range(900, 940)) + [2108, 3030, 3042])
def test_route_refine_random_small(seed):
    """Random small placements (1 to 4 copies per expert, 1 or 2 ranks per
    node, explicit sources, top-1 to top-4, C from 0 to 1).  Seeds 2108,
    3030 and 3042 have a source whose greedy result would raise its pairs,
    so it keeps its input routing."""
    rng = np.random.default_rng(seed)
    R = int(rng.choice([4, 6, 8]))
    rpn = int(rng.choice([1, 2]))
    E = int(rng.integers(3, 9))
    k = int(rng.integers(1, min(E, 4) + 1))
    T = int(rng.integers(1, 200))
    hosts = [sorted(rng.choice(R, size=int(rng.integers(1, 5)), replace=False).tolist())
             for _ in range(E)]
    src = rng.integers(0, R, size=T).astype(np.int32)
    pl = wl.placement_from_hosts(E, R, rpn, hosts, token_src_rank=src)
    ids_np = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)], dtype=np.int32)
    ids = torch.tensor(ids_np, device="cuda")
    c = (int(rng.integers(0, 3)), 2)
    slot, _, pl_dev, ws = _gpu_route_replicas(ids, pl, c)
    ref_in, _ = oracle.route_replicas_waterfill(ids_np, pl, *c)
    assert np.array_equal(slot.cpu().numpy(), ref_in)
    ref_slot, before, after = oracle.refine_consolidate(ids_np, ref_in, pl)
    slot, msgs = _gpu_refine(ids, pl_dev, slot, ws)
    assert np.array_equal(slot.cpu().numpy(), ref_slot) and msgs == (before, after)


@pytest.mark.parametrize("seed", range(6))
def test_route_refine_many_nodes_and_repeated_ids(seed):
    """The kernel's general path: more than 32 nodes (40 ranks of one GPU
    each), and tokens that name an expert twice (top-k ids are normally
    distinct; the refinement still follows the oracle's order there)."""
    rng = np.random.default_rng(4000 + seed)
    R, rpn, E, k, T = 40, 1, 6, 3, 3000
    hosts = [sorted(rng.choice(R, size=int(rng.integers(2, 5)), replace=False).tolist())
             for _ in range(E)]
    src = rng.integers(0, R, size=T).astype(np.int32)
    pl = wl.placement_from_hosts(E, R, rpn, hosts, token_src_rank=src)
    ids_np = np.array([rng.choice(E, size=k, replace=bool(seed % 2)) for _ in range(T)],
                      dtype=np.int32)
    ids = torch.tensor(ids_np, device="cuda")
    slot, _, pl_dev, ws = _gpu_route_replicas(ids, pl, (1, 2))
    ref_in, _ = oracle.route_replicas_waterfill(ids_np, pl, 1, 2)
    assert np.array_equal(slot.cpu().numpy(), ref_in)
    ref_slot, before, after = oracle.refine_consolidate(ids_np, ref_in, pl)
    slot, msgs = _gpu_refine(ids, pl_dev, slot, ws)
    assert np.array_equal(slot.cpu().numpy(), ref_slot) and msgs == (before, after)


def test_routed_layer_output_equals_fixed_rule_output():
    """Copies of an expert hold the same weights and rows are independent,
    so choosing other copies must not change the layer's output bit."""
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = wl.WORKLOADS["replica"].scaled(T=4096)
    pl = wl.make_placement(w)
    logits, x = wl.make_logits(w, "cuda"), wl.make_x(w, "cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    outs = []
    for relax in (None, (1, 10)):
        layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl),
                         w_gate_up=wgu, w_down=wd, max_tokens=w.T, replica_relax=relax)
        y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        layer.forward(logits, x, y)
        layer.check()
        outs.append((y, layer.rank_counts.clone(), int(layer.inter_node.item())))
    assert torch.equal(outs[0][0], outs[1][0])
    assert int(outs[0][1].sum()) == int(outs[1][1].sum()) == w.A


# ------------------------------------------------------------------ gather-fused FFN (no permute)
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "group_limited", "replica"])
def test_gather_layer_is_bit_identical_to_permuted_layer(name):
    """Reading the FFN's rows straight from x through the inverse
    permutation (TMA gather) must reproduce the permuted path bit for bit:
    h, the expert outputs and the layer output."""
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = wl.WORKLOADS[name]
    if name == "group_limited":
        w = w.scaled(T=1024)
    pl = wl.make_placement(w)
    logits, x = wl.make_logits(w, "cuda"), wl.make_x(w, "cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    sgu, sd = wl.make_shared_weights(w, "cuda")
    res = []
    for gather in (False, True):
        layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl),
                         w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                         n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                         shared_w_gate_up=sgu, shared_w_down=sd, gather=gather)
        y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        layer.forward(logits, x, y)
        layer.check()
        res.append((layer.h[:w.A].clone(), layer.y_perm[:w.A].clone(), y))
        del layer
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)


def test_gather_ffn_ragged_segments_match_oracle():
    """Small ragged case compared in full with the oracle, rows read through
    a shuffled inverse permutation."""
    m = moe()
    H, I, k, T = 512, 384, 2, 400
    counts = [130, 1, 0, 257, 128, 75, 209]
    E = len(counts) + 1
    w = wl.Workload("gath", 77, T=T, H=H, E=E, k=k, I=I, R=1, ranks_per_node=1)
    A = sum(counts)
    assert A == T * k
    g = torch.Generator(device="cuda").manual_seed(17)
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    src = torch.randperm(A, generator=g, device="cuda").to(torch.int32)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    se = torch.tensor([(3 * s + 1) % E for s in range(len(counts))], dtype=torch.int32, device="cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    h = torch.empty(A, I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(A, H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, len(counts))
    m.moe_grouped_ffn_gather(x, k, src, offs, se, pgu, pd, h, y, ws)
    m.moe_check_device_status(ws)
    rows = f64(x)[src.cpu().numpy() // k]
    rh, ry = oracle.grouped_ffn(rows, offs.cpu().numpy(), se.cpu().numpy(),
                                oracle.bf16_bits_to_f64(bits(wgu)), oracle.bf16_bits_to_f64(bits(wd)), I)
    assert_close(f64(h), rh, "h (gather)")
    assert_close(f64(y), ry, "y_perm (gather)")


def test_ffn_tile_size_boundaries_match_oracle_and_gather_bits():
    """Segments around the M = 64 rule (a tile runs M = 64 when at most 64
    rows remain in its segment): 1, 16, 63, 64, 65, 127, 128 and 129 rows,
    192 (a last block of exactly 64 rows), 193 (of 65) and 320.  Compared in
    full with the oracle, and bit for bit with the gather path, whose tiles
    are always 128 rows: a row's bits must not depend on the tile's M."""
    m = moe()
    H, I = 512, 256
    counts = [1, 16, 63, 64, 65, 127, 128, 129, 192, 193, 320]
    E = len(counts) + 1
    A = sum(counts)
    w = wl.Workload("m64", 81, T=A, H=H, E=E, k=1, I=I, R=1, ranks_per_node=1)
    g = torch.Generator(device="cuda").manual_seed(23)
    x = torch.randn(A, H, generator=g, device="cuda").to(torch.bfloat16)
    src = torch.arange(A, dtype=torch.int32, device="cuda")   # row r reads token r
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    se = torch.tensor([(5 * s + 3) % E for s in range(len(counts))], dtype=torch.int32, device="cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    ws = m.new_workspace(1, 1, len(counts))
    outs = []
    for gather in (False, True):
        h = torch.full((A, I), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = torch.full((A, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        if gather:
            m.moe_grouped_ffn_gather(x, 1, src, offs, se, pgu, pd, h, y, ws)
        else:
            m.moe_grouped_ffn_packed(x, offs, se, pgu, pd, h, y, ws)
        m.moe_check_device_status(ws)
        outs.append((h, y))
    rh, ry = oracle.grouped_ffn(f64(x), offs.cpu().numpy(), se.cpu().numpy(),
                                oracle.bf16_bits_to_f64(bits(wgu)), oracle.bf16_bits_to_f64(bits(wd)), I)
    assert_close(f64(outs[0][0]), rh, "h")
    assert_close(f64(outs[0][1]), ry, "y_perm")
    assert_ulps(f64(outs[0][0]), rh, "h", H_WITHIN1, H_BIG_MOST)
    assert_ulps(f64(outs[0][1]), ry, "y_perm", Y_WITHIN1, Y_BIG_MOST)
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


# ------------------------------------------------------------------ merge: node-local pre-reduction
@pytest.mark.parametrize("name", ["decode", "group_limited", "replica"])
def test_combine_merged_bit_exact_and_message_counts(name):
    m = moe()
    w = wl.WORKLOADS[name]
    if name == "group_limited":
        w = w.scaled(T=1024, H=1024)
    pl = wl.make_placement(w)
    pl_dev = m.DevicePlacement.from_tables(pl)
    ids, wts = gpu_route(w, wl.make_logits(w, "cuda"))
    lay = gpu_layout(ids, pl_dev, w.T, w.k)
    g = torch.Generator(device="cuda").manual_seed(w.index)
    yp = torch.randn(w.A, w.H, generator=g, device="cuda").to(torch.bfloat16)
    sh = torch.randn(w.T, w.H, generator=g, device="cuda").to(torch.bfloat16) if w.shared_I else None
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    msgs = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    dr = torch.from_numpy(lay["dest_row"]).cuda()
    slot = torch.from_numpy(lay["slot"]).cuda()
    m.moe_combine_merged(yp, dr, wts, slot, pl_dev, y, msgs, ws, sh)
    m.moe_check_device_status(ws)
    node = pl.slot_rank[lay["slot"]] // pl.ranks_per_node
    ref = oracle.combine_merged_fma32(bits(yp), lay["dest_row"], wts.cpu().numpy(), node,
                                      None if sh is None else bits(sh))
    assert np.array_equal(bits(y), ref)
    assert tuple(msgs.tolist()) == oracle.dispatch_messages(lay["slot"], pl, w.T, w.k)


def test_combine_merged_figure4_counts():
    m = moe()
    pl = wl.placement_from_hosts(3, 2, 1, [[1], [1], [0]], token_src_rank=np.array([0]))
    pl_dev = m.DevicePlacement.from_tables(pl)
    ids = torch.tensor([[0, 1, 2]], dtype=torch.int32, device="cuda")
    lay = gpu_layout(ids, pl_dev, 1, 3)
    yp = torch.ones(3, 8, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(1, 8, dtype=torch.bfloat16, device="cuda")
    msgs = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = m.new_workspace(1, 3, pl.n_slots)
    m.moe_combine_merged(yp, torch.from_numpy(lay["dest_row"]).cuda(),
                         torch.full((1, 3), 0.25, device="cuda"),
                         torch.from_numpy(lay["slot"]).cuda(), pl_dev, y, msgs, ws)
    m.moe_check_device_status(ws)
    assert msgs.tolist() == [2, 1]
    assert torch.equal(y.float(), torch.full((1, 8), 0.75, device="cuda"))


# ------------------------------------------------------------------ whole step as a CUDA graph
@pytest.mark.parametrize("name", ALL)
def test_weight_prefetch_is_only_a_hint(name):
    """moe_prefetch_ffn_weights derives the grouped FFN's first-wave tiles
    from the routed ids and asks L2 for their weights: it runs cleanly on
    every workload's routing and placement (full-size packed weights, so
    every fetched address is in bounds), and where the layer uses it (small
    dispatches: tiny, decode) the output bits are those of a step without it."""
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = wl.WORKLOADS[name]
    pl = wl.make_placement(w)
    dp = m.DevicePlacement.from_tables(pl)
    logits = wl.make_logits(w, "cuda")
    ids = torch.empty(w.T, w.k, dtype=torch.int32, device="cuda")
    tw = torch.empty(w.T, w.k, dtype=torch.float32, device="cuda")
    ws = m.new_workspace(w.T, w.k, dp.n_slots)
    m.moe_route(logits, route_cfg(w), ids, tw, ws)
    wgu = torch.empty(w.E, 2 * w.I, w.H, dtype=torch.bfloat16, device="cuda")
    m.moe_prefetch_ffn_weights(ids, dp, wgu, w.H, w.I, 64 << 20)
    torch.cuda.synchronize()
    m.moe_check_device_status(ws)
    del wgu
    if w.T * w.k * w.H * 2 > MoELayer.PREFETCH_MAX_DISPATCH:
        return
    x = wl.make_x(w, "cuda")
    layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=dp,
                     w_gate_up=wl.make_w_gate_up(w, "cuda"), w_down=wl.make_w_down(w, "cuda"),
                     max_tokens=w.T, score_fn=w.score_fn, n_groups=w.n_groups,
                     topk_groups=w.topk_groups, group_topn=w.group_topn)
    assert layer.prefetch_bytes > 0
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(logits, x, y)
    with_prefetch = y.clone()
    layer.prefetch_bytes = 0
    y.zero_()
    layer.forward(logits, x, y)
    torch.cuda.synchronize()
    layer.check()
    assert torch.equal(y, with_prefetch)


@pytest.mark.parametrize("name", ["decode", "group_limited", "replica"])
def test_graph_replay_matches_eager(name):
    """The step records into one CUDA graph (cooperative FFN, programmatic
    dependent launches, memsets) and its replays reproduce the eager step
    bit for bit, including after the inputs change in place."""
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    w = wl.WORKLOADS[name]
    if name == "group_limited":
        w = w.scaled(T=512, E=64, R=16, H=1024, I=256, shared_I=256)
    pl = wl.make_placement(w)
    logits, x = wl.make_logits(w, "cuda"), wl.make_x(w, "cuda")
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    sgu, sd = wl.make_shared_weights(w, "cuda")
    layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl),
                     w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                     n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                     shared_w_gate_up=sgu, shared_w_down=sd)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(logits, x, y)
    eager = y.clone()
    graph = layer.capture(logits, x, y)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    layer.check()
    assert torch.equal(y, eager)
    # new inputs in the same buffers: replay equals a fresh eager step
    g = torch.Generator(device="cuda").manual_seed(99)
    logits.copy_(torch.randn(logits.shape, generator=g, device="cuda"))
    x.copy_(torch.randn(x.shape, generator=g, device="cuda").to(torch.bfloat16))
    graph.replay()
    y_graph = y.clone()
    layer.forward(logits, x, y)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y)
