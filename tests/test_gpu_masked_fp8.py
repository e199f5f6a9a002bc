"""GPU parity of the fixed-capacity ("masked") layout and of FP8 dispatch,
through the C ABI, against the CPU oracle.

Bit-exact: the masked layout's every output (slots, demand, used rows,
rows, inverse, per-rank rows, drop count), the rows it moves, the combine
with dropped assignments, the E4M3 codes and block scales, the restored
bf16 rows.  The FFN on a masked layout is bit-identical to the contiguous
FFN on the same rows and within the FFN tolerance of the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from test_gpu_parity import (_BitsExperts, _LazyExperts, assert_close, bits, f64, gpu_route,
                             moe, oracle_route)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_ffn_gb300 import build
    build.build()
    oracle.build_c()
    torch.cuda.set_device(0)


def gpu_layout_masked(ids, pl_dev, T, k, cap, ws=None):
    m = moe()
    A, S = T * k, pl_dev.n_slots
    if ws is None:
        ws = m.new_workspace(T, k, S)
    i32 = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
    out = dict(slot=i32(A), seg_counts=i32(S), masked_m=i32(S), dest_row=i32(A),
               src_assign=i32(S * cap), rank_counts=i32(pl_dev.n_ranks), n_dropped=i32(1))
    m.moe_dispatch_layout_masked(ids, pl_dev, cap, out["slot"], out["seg_counts"], out["masked_m"],
                                 out["dest_row"], out["src_assign"], out["rank_counts"],
                                 out["n_dropped"], ws)
    m.moe_check_device_status(ws)
    res = {k_: v.cpu().numpy() for k_, v in out.items()}
    res["n_dropped"] = int(res["n_dropped"][0])
    return res


def assert_layout_equal(got, ref):
    for key in ("slot", "seg_counts", "masked_m", "dest_row", "src_assign", "rank_counts"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["n_dropped"] == ref["n_dropped"]


# ------------------------------------------------------------------ masked layout
@pytest.mark.parametrize("name,cap", [("tiny", 1), ("tiny", 16), ("decode", 2), ("decode", 64),
                                      ("prefill", 100), ("prefill", 4000), ("replica", 2000),
                                      ("group_limited", 96)])
def test_masked_layout_parity(name, cap):
    w = wl.WORKLOADS[name]
    m = moe()
    pl = wl.make_placement(w)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    got = gpu_layout_masked(ids, m.DevicePlacement.from_tables(pl), w.T, w.k, cap)
    ref = oracle.dispatch_layout_masked(ids.cpu().numpy(), pl, cap)
    assert_layout_equal(got, ref)


def test_masked_layout_drops_across_many_tiles_and_ragged_tail():
    """Several 1024-assignment tiles and a ragged last one, with a capacity
    small enough that drops happen in every tile: which assignments keep a
    row must follow assignment order across tile boundaries."""
    m = moe()
    w = wl.WORKLOADS["replica"].scaled(T=9000, k=3)
    pl = wl.make_placement(w)
    g = torch.Generator(device="cuda").manual_seed(5)
    ids = torch.stack([torch.randperm(w.E, generator=g, device="cuda")[:w.k] for _ in range(w.T)])
    ids = ids.to(torch.int32).contiguous()
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    for cap in (7, 300, 1000):
        got = gpu_layout_masked(ids, m.DevicePlacement.from_tables(pl), w.T, w.k, cap, ws)
        ref = oracle.dispatch_layout_masked(ids.cpu().numpy(), pl, cap)
        assert_layout_equal(got, ref)
        assert ref["n_dropped"] > 0 or cap == 1000


def test_masked_layout_worked_example():
    """The capacity example of "Capacity, padding, and the drop decision"
    (counts 22, 14, 7, 6, 5, 4, 3, 3; capacity 10) on the GPU."""
    m = moe()
    counts = [22, 14, 7, 6, 5, 4, 3, 3]
    pl = wl.placement_from_hosts(8, 8, 8, [[e] for e in range(8)])
    ids_np = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    ids_np = np.random.default_rng(1).permutation(ids_np).reshape(-1, 1).astype(np.int32)
    ids = torch.from_numpy(ids_np).cuda()
    got = gpu_layout_masked(ids, m.DevicePlacement.from_tables(pl), 64, 1, 10)
    assert_layout_equal(got, oracle.dispatch_layout_masked(ids_np, pl, 10))
    assert got["seg_counts"][0] - got["masked_m"][0] == 12
    assert got["rank_counts"].sum() == 64 - got["n_dropped"]


def test_masked_layout_leaves_workspace_clean_for_contiguous_layout():
    """The masked call clears the scan's flags like the contiguous one, so
    the two can alternate on one workspace."""
    from test_gpu_parity import gpu_layout
    m = moe()
    w = wl.WORKLOADS["prefill"]
    pl = wl.make_placement(w)
    pl_dev = m.DevicePlacement.from_tables(pl)
    ids, _ = gpu_route(w, wl.make_logits(w, "cuda"))
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    ids_np = ids.cpu().numpy()
    for _ in range(2):
        assert_layout_equal(gpu_layout_masked(ids, pl_dev, w.T, w.k, 150, ws),
                            oracle.dispatch_layout_masked(ids_np, pl, 150))
        lay = gpu_layout(ids, pl_dev, w.T, w.k, ws)
        assert np.array_equal(lay["dest_row"], oracle.dispatch_layout(ids_np, pl)["dest_row"])


# ------------------------------------------------------------------ permute / combine with drops
@pytest.mark.parametrize("name,cap", [("decode", 2), ("prefill", 120)])
def test_permute_and_combine_masked_bit_exact(name, cap):
    m = moe()
    w = wl.WORKLOADS[name]
    pl = wl.make_placement(w)
    ids, wts = gpu_route(w, wl.make_logits(w, "cuda"))
    lay = oracle.dispatch_layout_masked(ids.cpu().numpy(), pl, cap)
    assert lay["n_dropped"] > 0
    rows = pl.n_slots * cap
    x = wl.make_x(w, "cuda")
    dr = torch.from_numpy(lay["dest_row"]).cuda()
    xp = torch.full((rows, w.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(w.T, w.k, pl.n_slots)
    m.moe_permute_masked(x, w.k, dr, xp, ws)
    m.moe_check_device_status(ws)   # -1 rows are drops, not errors
    used = lay["src_assign"] >= 0
    ref = oracle.permute(bits(x), lay["dest_row"], w.k, n_rows=rows)
    assert np.array_equal(bits(xp)[used], ref[used])
    assert torch.isnan(xp[torch.from_numpy(~used).cuda()].float()).all()   # padding untouched
    g = torch.Generator(device="cuda").manual_seed(w.index)
    yp = torch.randn(rows, w.H, generator=g, device="cuda").to(torch.bfloat16)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    m.moe_combine_masked(yp, dr, wts, y, ws)
    m.moe_check_device_status(ws)
    assert np.array_equal(bits(y), oracle.combine_fma32(bits(yp), lay["dest_row"], wts.cpu().numpy()))


def test_plain_combine_still_reports_a_dropped_row():
    """Only the masked entry points accept -1; the contiguous combine keeps
    treating it as an index error."""
    m = moe()
    T, k, H = 4, 2, 64
    yp = torch.ones(T * k, H, dtype=torch.bfloat16, device="cuda")
    dr = torch.arange(T * k, dtype=torch.int32, device="cuda")
    dr[3] = -1
    y = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(T, k, 1)
    m.moe_combine(yp, dr, torch.ones(T, k, device="cuda"), y, ws)
    with pytest.raises(m.MoeError) as ei:
        m.moe_check_device_status(ws)
    assert ei.value.status == 4


# ------------------------------------------------------------------ grouped FFN on the masked layout
@pytest.mark.parametrize("H,I,cap,used", [(256, 128, 5, [3, 0, 5, 1]),
                                          (512, 384, 300, [130, 1, 0, 257, 300, 75]),
                                          (256, 256, 128, [128, 127, 0])])
def test_masked_ffn_matches_oracle_and_contiguous_ffn(H, I, cap, used):
    m = moe()
    S = len(used)
    E = S + 1
    w = wl.Workload("ffnm", 90 + H // 256 + I + cap, T=1, H=H, E=E, k=1, I=I, R=1,
                    ranks_per_node=1)
    rows = S * cap
    g = torch.Generator(device="cuda").manual_seed(cap)
    xp = torch.randn(rows, H, generator=g, device="cuda").to(torch.bfloat16)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    se = torch.tensor([(2 * s + 1) % E for s in range(S)], dtype=torch.int32, device="cuda")
    mm = torch.tensor(used, dtype=torch.int32, device="cuda")
    h = torch.full((rows, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((rows, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, S)
    m.moe_grouped_ffn_masked(xp, cap, mm, se, pgu, pd, h, y, ws)
    m.moe_check_device_status(ws)
    keep = np.concatenate([s * cap + np.arange(used[s]) for s in range(S)])
    rh, ry = oracle.grouped_ffn_masked(f64(xp), cap, np.array(used), se.cpu().numpy(),
                                       oracle.bf16_bits_to_f64(bits(wgu)),
                                       oracle.bf16_bits_to_f64(bits(wd)), I)
    kt = torch.from_numpy(keep).cuda()
    assert_close(f64(h[kt]), rh[keep], "h (masked)")
    assert_close(f64(y[kt]), ry[keep], "y_perm (masked)")
    pad = torch.from_numpy(np.setdiff1d(np.arange(rows), keep)).cuda()
    assert torch.isnan(y[pad].float()).all() and torch.isnan(h[pad].float()).all()
    # the same rows packed contiguously give the same bits
    offs = torch.tensor(np.concatenate([[0], np.cumsum(used)]), dtype=torch.int32, device="cuda")
    xc = xp[kt].contiguous()
    hc = torch.empty(len(keep), I, dtype=torch.bfloat16, device="cuda")
    yc = torch.empty(len(keep), H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_ffn_packed(xc, offs, se, pgu, pd, hc, yc, ws)
    m.moe_check_device_status(ws)
    assert torch.equal(hc, h[kt]) and torch.equal(yc, y[kt])


def test_masked_ffn_reports_a_count_above_capacity():
    m = moe()
    w = wl.Workload("ffnx", 95, T=1, H=256, E=2, k=1, I=128, R=1, ranks_per_node=1)
    wgu, wd = wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda")
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    m.moe_pack_expert_weights(wgu, wd, pgu, pd)
    cap = 4
    xp = torch.zeros(2 * cap, 256, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(2 * cap, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(2 * cap, 256, dtype=torch.bfloat16, device="cuda")
    ws = m.new_workspace(1, 1, 2)
    m.moe_grouped_ffn_masked(xp, cap, torch.tensor([2, 9], dtype=torch.int32, device="cuda"),
                             torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                             pgu, pd, h, y, ws)
    with pytest.raises(m.MoeError) as ei:
        m.moe_check_device_status(ws)
    assert ei.value.status == 4
    # segment 1 clamped to cap: all its rows computed (zero in, zero out);
    # segment 0's two rows computed, its padding left alone
    assert torch.equal(y[:2], torch.zeros_like(y[:2]))
    assert torch.equal(y[cap:], torch.zeros_like(y[cap:]))


# ------------------------------------------------------------------ whole layer, masked
def _layer(w, pl, wgu, wd, sgu, sd, **kw):
    from grouped_ffn_gb300 import MoELayer
    m = moe()
    return MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=m.DevicePlacement.from_tables(pl),
                    w_gate_up=wgu, w_down=wd, max_tokens=w.T, score_fn=w.score_fn,
                    n_groups=w.n_groups, topk_groups=w.topk_groups, group_topn=w.group_topn,
                    shared_w_gate_up=sgu, shared_w_down=sd, **kw)


def _inputs(w):
    return (wl.make_placement(w), wl.make_logits(w, "cuda"), wl.make_x(w, "cuda"),
            wl.make_w_gate_up(w, "cuda"), wl.make_w_down(w, "cuda"),
            *wl.make_shared_weights(w, "cuda"))


@pytest.mark.parametrize("name", ["decode", "replica"])
def test_masked_layer_without_drops_equals_contiguous_layer(name):
    w = wl.WORKLOADS[name]
    if name == "replica":
        w = w.scaled(T=2048)
    pl, logits, x, wgu, wd, sgu, sd = _inputs(w)
    outs = []
    for cap in (None, w.T):
        layer = _layer(w, pl, wgu, wd, sgu, sd, masked_cap=cap)
        y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        layer.forward(logits, x, y)
        layer.check()
        outs.append((y, layer.rank_counts.clone(), layer.balancedness.clone()))
        if cap is not None:
            assert layer.n_dropped.item() == 0
        del layer
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])


def test_masked_layer_with_drops_matches_oracle():
    """Capacity 1.25x the mean load: hot experts drop assignments.  Layout
    bit-exact; the combine bit-exact from the GPU's expert outputs; sampled
    tokens against the layer's definition with the dropped experts' terms
    removed.  Decode routing and token count at a narrower width, so that
    the definition can be evaluated for every token."""
    w = wl.WORKLOADS["decode"].scaled(H=1024, I=512)
    pl, logits, x, wgu, wd, sgu, sd = _inputs(w)
    cap = int(1.25 * w.A / pl.n_slots) + 1
    layer = _layer(w, pl, wgu, wd, sgu, sd, masked_cap=cap)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(logits, x, y)
    layer.check()
    ids_ref, _, _ = oracle_route(w, logits.cpu().numpy())
    lay = oracle.dispatch_layout_masked(ids_ref, pl, cap)
    assert lay["n_dropped"] > 0 and layer.n_dropped.item() == lay["n_dropped"]
    assert np.array_equal(layer.dest_row[:w.A].cpu().numpy(), lay["dest_row"])
    assert np.array_equal(layer.masked_m.cpu().numpy(), lay["masked_m"])
    assert np.array_equal(layer.rank_counts.cpu().numpy(), lay["rank_counts"])
    ref_y = oracle.combine_fma32(bits(layer.y_perm), lay["dest_row"], layer.topk_w[:w.T].cpu().numpy())
    assert np.array_equal(bits(y), ref_y)
    # used rows of the FFN against the oracle
    keep = np.nonzero(lay["src_assign"] >= 0)[0]
    kt = torch.from_numpy(keep).cuda()
    full = np.zeros((pl.n_slots * cap, w.H))
    full[keep] = f64(layer.x_perm[kt])
    _, ry = oracle.grouped_ffn_masked(full, cap, lay["masked_m"], pl.slot_expert,
                                      _LazyExperts(wgu), _LazyExperts(wd), w.I)
    assert_close(f64(layer.y_perm[kt]), ry[keep], "y_perm (masked layer)")
    # tokens from the definition, dropped experts removed
    toks = np.arange(w.T)
    xr = f64(x)
    wts = layer.topk_w[:w.T].cpu().numpy().astype(np.float64)
    ref = np.zeros((w.T, w.H))
    gu, dd = _LazyExperts(wgu), _LazyExperts(wd)
    for t in toks:
        acc = np.zeros(w.H)
        for j in range(w.k):
            if lay["dest_row"][t * w.k + j] < 0:
                continue
            _, ye = oracle.swiglu_expert(xr[t][None, :], gu[int(ids_ref[t, j])], dd[int(ids_ref[t, j])], w.I)
            acc = acc + wts[t, j] * ye[0]
        ref[t] = oracle.bf16_round(acc)
    assert_close(f64(y), ref, "masked layer output")


def test_masked_graph_replay_matches_eager():
    """One graph for the fixed-capacity step; replays after the routing
    changes give what a fresh eager step gives."""
    w = wl.WORKLOADS["decode"]
    pl, logits, x, wgu, wd, sgu, sd = _inputs(w)
    layer = _layer(w, pl, wgu, wd, sgu, sd, masked_cap=48)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(logits, x, y)
    eager = y.clone()
    graph = layer.capture(logits, x, y)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    layer.check()
    assert torch.equal(y, eager)
    g = torch.Generator(device="cuda").manual_seed(7)
    logits.copy_(torch.randn(logits.shape, generator=g, device="cuda") * 3)
    graph.replay()
    torch.cuda.synchronize()
    replayed = y.clone()
    layer.forward(logits, x, y)
    torch.cuda.synchronize()
    layer.check()
    assert torch.equal(replayed, y)


# ------------------------------------------------------------------ FP8 dispatch
def _special_x(T, H, seed):
    """bf16 rows whose 128-channel blocks cover the scale rule's cases: all
    zero, signed zeros, a maximum exactly 448 and just above, bf16
    subnormals, values near the top of the bf16 range, and plain N(0,1)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(T, H, generator=g)
    nb = H // 128
    for t in range(T):
        b = t % nb
        blk = slice(b * 128, (b + 1) * 128)
        kind = t % 7
        if kind == 0:
            x[t, blk] = 0.0
        elif kind == 1:
            x[t, blk] = -0.0
        elif kind == 2:
            x[t, blk] *= 100.0
            x[t, b * 128] = 448.0
        elif kind == 3:
            x[t, b * 128 + 5] = -450.0
        elif kind == 4:
            x[t, blk] *= 1e-39               # bf16 subnormals
        elif kind == 5:
            x[t, blk] = x[t, blk].clamp(-1, 1) * 3.0e38
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,H,k", [(70, 256, 2), (333, 1024, 4), (64, 8192, 2)])
def test_permute_fp8_codes_and_scales_bit_exact(T, H, k):
    m = moe()
    x = _special_x(T, H, T + H).cuda()
    g = torch.Generator(device="cpu").manual_seed(T)
    dr_np = torch.randperm(T * k, generator=g).numpy().astype(np.int32)
    dr_np[::11] = -1                       # a few drops
    dr = torch.from_numpy(dr_np).cuda()
    n = T * k
    xq = torch.full((n, H), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((n, H // 128), -1.0, device="cuda")
    ws = m.new_workspace(T, k, 1)
    m.moe_permute_fp8(x, k, dr, xq, xs, ws)
    m.moe_check_device_status(ws)
    codes, scales = oracle.quantize_fp8_blocks(bits(x))
    got_q, got_s = xq.cpu().numpy(), xs.cpu().numpy()
    for a in range(n):
        r = dr_np[a]
        if r < 0:
            continue
        assert np.array_equal(got_q[r], codes[a // k]), f"codes of assignment {a}"
        assert np.array_equal(got_s[r], scales[a // k]), f"scales of assignment {a}"
    unused = np.setdiff1d(np.arange(n), dr_np[dr_np >= 0])
    assert np.all(got_q[unused] == 0xAB) and np.all(got_s[unused] == -1.0)


@pytest.mark.parametrize("masked", [False, True])
def test_dequant_fp8_bit_exact(masked):
    m = moe()
    H, S, cap = 1024, 5, 40
    n = S * cap
    g = torch.Generator(device="cpu").manual_seed(11)
    codes = torch.randint(0, 256, (n, H), generator=g, dtype=torch.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11    # no NaN codes
    e = torch.randint(-126, 100, (n, H // 128), generator=g)
    e[0, 0], e[1, 0] = -126, 127 - 9       # the clamp's end and a large scale
    scales = torch.pow(2.0, e.double()).float()
    mm = torch.tensor([0, 40, 17, 1, 39], dtype=torch.int32)
    out = torch.full((n, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.moe_dequant_fp8(codes.cuda(), scales.cuda(), out, mm.cuda() if masked else None,
                      cap if masked else 0)
    torch.cuda.synchronize()
    ref = oracle.dequantize_fp8_blocks(codes.numpy(), scales.numpy())
    got = bits(out)
    if masked:
        used = np.concatenate([s * cap + np.arange(int(mm[s])) for s in range(S)])
        assert np.array_equal(got[used], ref[used])
        pad = np.setdiff1d(np.arange(n), used)
        assert torch.isnan(out[torch.from_numpy(pad).cuda()].float()).all()
    else:
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("name,cap", [("decode", None), ("prefill", None), ("decode", 20)])
def test_fp8_dispatch_layer(name, cap):
    """Layer with FP8 dispatch: the restored rows equal the oracle's
    quantize-then-restore of x, bit for bit; the FFN on them and the
    combine match the oracle as in the bf16 layer."""
    w = wl.WORKLOADS[name]
    pl, logits, x, wgu, wd, sgu, sd = _inputs(w)
    layer = _layer(w, pl, wgu, wd, sgu, sd, fp8_dispatch=True, masked_cap=cap)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(logits, x, y)
    layer.check()
    ids_ref, _, _ = oracle_route(w, logits.cpu().numpy())
    lay = (oracle.dispatch_layout(ids_ref, pl) if cap is None
           else oracle.dispatch_layout_masked(ids_ref, pl, cap))
    rng = np.random.default_rng(w.index)
    toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, size=min(40, w.T), replace=False)]))
    codes, scales = oracle.quantize_fp8_blocks(bits(x[torch.from_numpy(toks).cuda()]))
    restored = oracle.dequantize_fp8_blocks(codes, scales)
    for i, t in enumerate(toks):
        for j in range(w.k):
            r = lay["dest_row"][t * w.k + j]
            if r >= 0:
                assert np.array_equal(bits(layer.x_perm[r]), restored[i]), (t, j)
    # combine from the GPU's expert outputs, bit-exact
    ref_y = oracle.combine_fma32(bits(layer.y_perm), lay["dest_row"], layer.topk_w[:w.T].cpu().numpy())
    assert np.array_equal(bits(y), ref_y)
    # sampled tokens through the definition on the restored rows
    cfg = dict(score_fn=w.score_fn, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
               group_topn=w.group_topn)
    xq_bits = bits(x).copy()
    xq_bits[toks] = restored
    if cap is None:
        ref = oracle.moe_layer_tokens(toks, logits.cpu().numpy(), xq_bits, _BitsExperts(wgu),
                                      _BitsExperts(wd), pl, cfg, I=w.I)
        assert_close(f64(y[torch.from_numpy(toks).cuda()]), ref, "fp8-dispatch layer output")
    # the FP8 layer stays close to the bf16 layer (information, not parity)
    base = _layer(w, pl, wgu, wd, sgu, sd, masked_cap=cap)
    yb = torch.empty_like(y)
    base.forward(logits, x, yb)
    base.check()
    rel = (torch.linalg.norm(y.float() - yb.float()) / torch.linalg.norm(yb.float())).item()
    assert rel < 0.08, rel
