"""Pins of the oracle's fixed-capacity ("masked") layout and FP8 dispatch.

Masked layout: "14. Serving Mixture-of-Experts Models", "Capacity, padding,
and the drop decision" (its worked example, in tests/golden) and
"Mixture-of-Experts Inference", "Communication pressure" (decode pads
tokens into fixed-size masked layouts).  FP8: the same page and section
(activations quantized to FP8 before dispatch), with the OCP E4M3 format
checked against its bit-field definition, exhaustive round trips, hand
midpoints and PyTorch's own float8_e4m3fn conversion.  CPU only."""

import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "capacity_worked_example.json")


def _one_expert_per_rank(E):
    return wl.placement_from_hosts(E, E, 1, [[e] for e in range(E)])


def _ids_with_counts(counts, seed=0):
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    return np.random.default_rng(seed).permutation(ids).reshape(-1, 1)


# ---------------------------------------------------------------- masked layout
def test_worked_example_capacity_and_padding():
    g = json.load(open(GOLDEN))
    counts = g["expert_counts"]
    E = len(counts)
    assert sum(counts) == g["total_assignments"] == E * g["mean_per_expert"]
    pl = _one_expert_per_rank(E)
    ids = _ids_with_counts(counts)
    cf = g["capacity_factor"]
    assert cf["capacity"] == int(cf["factor"] * g["mean_per_expert"])
    lay = oracle.dispatch_layout_masked(ids, pl, cf["capacity"])
    assert E * cf["capacity"] == cf["rows"]
    e0 = cf["expert"]
    assert lay["seg_counts"][e0] - lay["masked_m"][e0] == cf["expert_overflow"]
    assert list(lay["masked_m"]) == [min(c, cf["capacity"]) for c in counts]
    assert list(lay["seg_counts"]) == counts
    assert lay["n_dropped"] == sum(max(0, c - cf["capacity"]) for c in counts)
    assert int((lay["dest_row"] < 0).sum()) == lay["n_dropped"]
    assert lay["rank_counts"].sum() + lay["n_dropped"] == g["total_assignments"]
    pm = g["pad_to_max"]
    assert max(counts) == pm["capacity"]
    lay = oracle.dispatch_layout_masked(ids, pl, pm["capacity"])
    assert lay["n_dropped"] == 0
    assert E * pm["capacity"] == pm["rows"]
    assert int((lay["src_assign"] >= 0).sum()) == pm["useful_rows"]
    frac = 1 - pm["useful_rows"] / pm["rows"]
    assert 0.6 < frac < 0.7            # "about two thirds" of the rows are padding


def _check_masked(ids, pl, cap):
    T, k = ids.shape
    A = T * k
    lay = oracle.dispatch_layout_masked(ids, pl, cap)
    S = pl.n_slots
    slot, dr, sa = lay["slot"], lay["dest_row"], lay["src_assign"]
    # the kept assignments of each slot are its first `cap` in assignment order
    for s in range(S):
        mine = np.nonzero(slot == s)[0]
        kept, dropped = mine[:cap], mine[cap:]
        assert np.array_equal(dr[kept], s * cap + np.arange(len(kept)))
        assert np.all(dr[dropped] == -1)
        assert np.array_equal(sa[s * cap:s * cap + len(kept)], kept)
        assert np.all(sa[s * cap + len(kept):(s + 1) * cap] == -1)
        assert int(pl.slot_expert[s]) == 0 or len(mine) == 0 or \
            np.all(ids.reshape(-1)[mine] == pl.slot_expert[s])
    assert np.array_equal(lay["seg_counts"], np.bincount(slot, minlength=S))
    assert np.array_equal(lay["masked_m"], np.minimum(lay["seg_counts"], cap))
    assert lay["n_dropped"] == int(np.maximum(lay["seg_counts"] - cap, 0).sum())
    assert lay["rank_counts"].sum() == A - lay["n_dropped"]
    return lay


def test_masked_layout_invariants_and_reduction_to_contiguous():
    w = wl.WORKLOADS["decode"]
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    for cap in (1, 2, 3, 5, w.T):
        lay = _check_masked(ids, pl, cap)
    # with room for everything the masked rows are the contiguous rows, moved
    cont = oracle.dispatch_layout(ids, pl)
    lay = _check_masked(ids, pl, w.T)
    assert lay["n_dropped"] == 0
    assert np.array_equal(lay["rank_counts"], cont["rank_counts"])
    off = cont["seg_offsets"]
    for a in range(w.A):
        s = int(cont["slot"][a])
        assert lay["dest_row"][a] - s * w.T == cont["dest_row"][a] - off[s]


def test_masked_layout_with_replicas_follows_the_slot_rule():
    w = wl.WORKLOADS["replica"].scaled(T=512)
    pl = wl.make_placement(w)
    ids, _ = oracle.route_softmax_topk(wl.make_logits(w).numpy(), w.k)
    lay = _check_masked(ids, pl, 40)
    cont = oracle.dispatch_layout(ids, pl)
    assert np.array_equal(lay["slot"], cont["slot"])


def test_dropped_assignment_contributes_zero():
    rng = np.random.default_rng(5)
    T, k, H, cap = 24, 2, 32, 3
    pl = _one_expert_per_rank(4)
    ids = np.stack([np.zeros(T, np.int32), rng.integers(1, 4, T).astype(np.int32)], 1)
    lay = oracle.dispatch_layout_masked(ids, pl, cap)
    assert lay["n_dropped"] > 0
    y_perm = oracle.bf16_round(rng.standard_normal((4 * cap, H)))
    w = rng.uniform(0.1, 1, (T, k)).astype(np.float32)
    # same as giving the dropped assignments weight zero on an all-kept layout
    dr = lay["dest_row"]
    w0 = w.copy().reshape(-1)
    w0[dr < 0] = 0.0
    dr_fill = np.where(dr < 0, 0, dr)
    got = oracle.combine_f64(y_perm, dr, w.astype(np.float64))
    ref = oracle.combine_f64(y_perm, dr_fill, w0.reshape(T, k).astype(np.float64))
    assert np.array_equal(got, ref)
    bits = oracle.f64_to_bf16_bits(y_perm)
    got32 = oracle.combine_fma32(bits, dr, w)
    ref32 = oracle.combine_fma32(bits, dr_fill, w0.reshape(T, k))
    f = oracle.bf16_bits_to_f64
    assert np.array_equal(f(got32), f(ref32))    # equal as values (+0 / -0 aside)
    # a token whose every assignment was dropped gets exactly the shared part
    sh = oracle.f64_to_bf16_bits(oracle.bf16_round(rng.standard_normal((T, H))))
    all_dropped = np.full(T * k, -1, np.int32)
    assert np.array_equal(oracle.combine_fma32(bits, all_dropped, w, sh), sh)


def test_permute_skips_dropped_rows():
    x = np.arange(6 * 4, dtype=np.uint16).reshape(6, 4)
    dr = np.array([4, -1, 0, 2, -1, 5, 1, 3, -1, -1, 6, 7], np.int32)
    out = oracle.permute(x, dr, 2, n_rows=8)
    for a, r in enumerate(dr):
        if r >= 0:
            assert np.array_equal(out[r], x[a // 2])


def test_masked_ffn_rows_equal_contiguous_ffn_rows():
    rng = np.random.default_rng(6)
    H, I, E, cap = 16, 8, 3, 5
    m = np.array([2, 0, 5], np.int32)
    xp = oracle.bf16_round(rng.standard_normal((3 * cap, H)))
    wgu = oracle.bf16_round(rng.standard_normal((E, 2 * I, H)) * 0.3)
    wd = oracle.bf16_round(rng.standard_normal((E, H, I)) * 0.3)
    seg_expert = np.array([2, 0, 1], np.int32)
    h, y = oracle.grouped_ffn_masked(xp, cap, m, seg_expert, wgu, wd, I)
    rows = np.concatenate([s * cap + np.arange(m[s]) for s in range(3)])
    off = np.concatenate([[0], np.cumsum(m)])
    hc, yc = oracle.grouped_ffn(xp[rows], off, seg_expert, wgu, wd, I)
    assert np.array_equal(h[rows], hc) and np.array_equal(y[rows], yc)
    pad = np.setdiff1d(np.arange(3 * cap), rows)
    assert np.all(y[pad] == 0)


# ---------------------------------------------------------------- E4M3
def test_e4m3_bit_fields():
    v = oracle.e4m3_value
    assert v(0x00) == 0.0 and np.signbit(v(0x80))
    assert v(0x01) == 2.0 ** -9                 # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert v(0x08) == 2.0 ** -6                 # smallest normal
    assert v(0x38) == 1.0                       # exponent field 7 = bias
    assert v(0x3C) == 1.5
    assert v(0x7E) == 448.0                     # largest finite
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0xC0) == -2.0
    pos = v(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)             # codes are ordered like values
    assert len(set(v(np.arange(256))[~np.isnan(v(np.arange(256)))])) == 253  # +0 == -0


def test_e4m3_encode_round_trip_and_ties():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_value(codes)), codes)
    enc = oracle.e4m3_encode
    assert enc(1.0625) == 0x38                  # halfway 1 .. 1.125 -> even (1.0)
    assert enc(1.1875) == 0x3A                  # halfway 1.125 .. 1.25 -> even (1.25)
    assert enc(2.0 ** -10) == 0x00              # halfway 0 .. 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02          # halfway 2^-9 .. 2^-8 -> even
    assert enc(-0.0) == 0x80 and enc(-1e-300) == 0x80
    assert enc(416.0) == 0x7D and enc(440.0) == 0x7E   # 416 = 1.625 * 2^8 exactly
    assert enc(400.0) == 0x7C and enc(408.0) == 0x7D   # 400: halfway 384 .. 416 -> even
    assert enc(1.0 + 2.0 ** -30) == 0x38 and enc(1.0625 + 2.0 ** -30) == 0x39
    with pytest.raises(ValueError):
        enc(449.0)


def test_e4m3_encode_matches_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000),
                        rng.standard_normal(2000) * 2.0 ** -7])
    v = v.astype(np.float32)       # exact in fp64 too
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_block_exponent():
    e = oracle.fp8_block_exponent
    assert e(448.0) == 0 and e(450.0) == 1 and e(896.0) == 1 and e(898.0) == 2
    assert e(1.0) == -8 and e(1.75) == -8 and e(1.7578125) == -7
    assert e(0.0) == 0
    assert e(2.0 ** -130) == -126               # clamped
    rng = np.random.default_rng(8)
    for a in np.abs(rng.standard_normal(200)) * 10.0 ** rng.uniform(-5, 5, 200):
        k = e(a)
        assert a <= 448 * 2.0 ** k and a > 448 * 2.0 ** (k - 1)


def test_quantize_blocks_bounds_and_exact_cases():
    rng = np.random.default_rng(9)
    x = oracle.bf16_round(rng.standard_normal((6, 256)) * np.array([[1e-3], [1], [30], [1], [1], [5e3]]))
    x[4] = 0.0
    bits = oracle.f64_to_bf16_bits(x)
    codes, scales = oracle.quantize_fp8_blocks(bits)
    assert codes.shape == (6, 256) and scales.shape == (6, 2)
    s64 = scales.astype(np.float64)
    assert np.all(np.log2(s64) == np.round(np.log2(s64)))     # powers of two
    vals = oracle.e4m3_value(codes)
    for t in range(6):
        for b in range(2):
            blk = vals[t, b * 128:(b + 1) * 128]
            amax = np.max(np.abs(blk))
            if t == 4:
                assert amax == 0 and scales[t, b] == 1.0
            else:
                assert 224 < amax <= 448   # the largest code uses the top binade
    back = oracle.bf16_bits_to_f64(oracle.dequantize_fp8_blocks(codes, scales))
    err = np.abs(back - x)
    scale_rep = np.repeat(s64, 128, axis=1)
    # nearest rounding: half a step of the 3-bit mantissa (relative 2^-4),
    # or half the subnormal step 2^-10 * scale, plus the bf16 rounding
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale_rep) * (1 + 2.0 ** -7)
    assert np.all(err <= bound)
    # values already on the E4M3 grid of their block come back unchanged
    grid = oracle.e4m3_value(rng.integers(0, 0x7F, (2, 128)).astype(np.uint8)) * 2.0 ** -3
    grid[:, 0] = 448 * 2.0 ** -3                # pin the block maximum, scale 2^-3
    gb = oracle.f64_to_bf16_bits(grid)
    c2, s2 = oracle.quantize_fp8_blocks(gb)
    assert np.all(s2 == np.float32(2.0 ** -3))
    assert np.array_equal(oracle.dequantize_fp8_blocks(c2, s2), gb)


def test_dequantize_rounds_bf16_subnormals_to_even():
    # code 0x01 (2^-9) * 2^-126 = 2^-135: a quarter of the bf16 subnormal
    # step 2^-133 -> 0; code 0x02 * 2^-126 = 2^-134 is a tie -> 0 (even);
    # code 0x06 * 2^-126 = 3 * 2^-134 is a tie between 2^-133 and 2^-132 -> 2^-132
    codes = np.zeros((1, 128), np.uint8)
    codes[0, :3] = [0x01, 0x02, 0x06]
    scales = np.array([[2.0 ** -126]], np.float32)
    got = oracle.bf16_bits_to_f64(oracle.dequantize_fp8_blocks(codes, scales))[0, :3]
    assert list(got) == [0.0, 0.0, 2.0 ** -132]
