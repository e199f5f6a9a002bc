"""The grouped FFN's tile schedule (moe_ffn_schedule, passed explicitly to
moe_grouped_ffn_packed_scheduled) changes how tiles are run, never the
arithmetic of a row: the layer's h, y_perm and y are bit-identical under
every setting.  ph1_shift (phase-1 positions given first to the CTAs with
one gate/up tile fewer) and interleave=0 (plain segment order) change which
CTA runs a tile and when; small_tiles=0 runs segments of at most 64 rows as
128-row tiles instead of M = 64 ones; cta_pairs=1 runs 256-row tiles on a pair
of SMs (tcgen05 cta_group::2) instead of 128-row tiles on one."""

import hashlib

import numpy as np

import pytest
import torch

pytestmark = pytest.mark.gpu


def _layer_hash(schedule):
    import workloads as wl
    from grouped_ffn_gb300 import MoELayer, moe
    dev = torch.device("cuda", 0)
    # 4000 tokens, top-2 over 64 experts with Zipf 1.0 skew and a shared
    # expert in the routed launch: over 100 m-blocks, so the gate/up phase
    # has more tiles than the 152 CTAs and a partial last wave that the shift
    # rebalances, and the skew's tail has many segments of at most 64 rows.
    w = wl.Workload("schedule", 91, T=4000, H=1024, E=64, k=2, I=512, R=8, ranks_per_node=8,
                    shared_I=512, zipf_s=1.0)
    pl = wl.make_placement(w)
    logits, x = wl.make_logits(w, dev), wl.make_x(w, dev)
    sgu, sd = wl.make_shared_weights(w, dev)
    layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k,
                     placement=moe.DevicePlacement.from_tables(pl, dev),
                     w_gate_up=wl.make_w_gate_up(w, dev), w_down=wl.make_w_down(w, dev),
                     max_tokens=w.T, shared_w_gate_up=sgu, shared_w_down=sd, device=dev,
                     ffn_schedule=schedule)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        layer.forward(logits, x, y, st)
    st.synchronize()
    layer.check(st)
    rows = w.A + w.T
    h = hashlib.sha256()
    for t in (layer.h[:rows], layer.y_perm[:rows], y):
        h.update(t.contiguous().view(torch.int16).cpu().numpy().tobytes())
    small = int(((layer.seg_counts > 0) & (layer.seg_counts <= 64)).sum().item())
    return h.hexdigest(), small


def test_tile_schedules_give_identical_bits():
    from grouped_ffn_gb300 import moe
    ref, small = _layer_hash(None)
    assert small >= 8, small   # the M = 64 path is exercised
    for sched in ((0, 1, 1, 1), (7, 1, 1, 1), (-1, 0, 1, 1), (0, 0, 1, 1), (-1, 1, 1, 1),
                  (-1, 1, 1, 0), (0, 1, 1, 0), (-1, 0, 1, 0), (-1, 1, 0, 0), (-1, 0, 0, 0)):
        assert _layer_hash(moe.FfnSchedule(*sched)) == (ref, small), sched


def test_schedule_arguments_are_checked():
    from grouped_ffn_gb300 import moe
    dev = torch.device("cuda", 0)
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device=dev)
    wgu = torch.zeros(1, 256, 256, dtype=torch.bfloat16, device=dev)
    wd = torch.zeros(1, 256, 128, dtype=torch.bfloat16, device=dev)
    offs = torch.tensor([0, 4], dtype=torch.int32, device=dev)
    ex = torch.zeros(1, dtype=torch.int32, device=dev)
    h = torch.empty(4, 128, dtype=torch.bfloat16, device=dev)
    y = torch.empty(4, 256, dtype=torch.bfloat16, device=dev)
    ws = moe.new_workspace(4, 1, 1, device=dev)
    for bad in ((-2, 1, 1, 1), (0, 2, 1, 1), (0, 1, -1, 1), (0, 1, 1, 2)):
        with pytest.raises(moe.MoeError):
            moe.moe_grouped_ffn_packed_scheduled(x, offs, ex, wgu, wd, 0, 0, 0,
                                                 moe.FfnSchedule(*bad), h, y, ws)


def test_ffn_leaves_its_counters_clear_for_the_next_call():
    """The grouped FFN runs with no memset before it: its per-segment
    readiness counters (workspace bytes [256, 256 + 4*S)) and its
    finished-CTA counter (status-block word 16) must be zero on entry, and
    the last CTA of each launch clears them.  Calls of different segment
    counts and tile counts, single-SM and SM-pair schedules, one after
    another on one workspace, each leave them zero and give the same bits
    as the same call on a fresh workspace."""
    from grouped_ffn_gb300 import moe
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(17)
    H, I, E = 512, 256, 12
    wgu = (torch.randn(E, 2 * I, H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    wd = (torch.randn(E, H, I, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    pgu, pd = torch.empty_like(wgu), torch.empty_like(wd)
    moe.moe_pack_expert_weights(wgu, wd, pgu, pd)
    ws = moe.new_workspace(4096, 2, 1024, device=dev)

    def run(counts, sched, ws_):
        offs = torch.zeros(len(counts) + 1, dtype=torch.int32)
        offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
        n = int(offs[-1])
        x = (torch.randn(n, H, generator=g, device=dev)).to(torch.bfloat16)
        ex = torch.tensor([i % E for i in range(len(counts))], dtype=torch.int32, device=dev)
        h = torch.empty(n, I, dtype=torch.bfloat16, device=dev)
        y = torch.empty(n, H, dtype=torch.bfloat16, device=dev)
        moe.moe_grouped_ffn_packed_scheduled(x, offs.to(dev), ex, pgu, pd, 0, 0, 0, sched, h, y, ws_)
        torch.cuda.synchronize()
        moe.moe_check_device_status(ws_)
        fresh = moe.new_workspace(4096, 2, 1024, device=dev)
        y2 = torch.empty_like(y)
        moe.moe_grouped_ffn_packed_scheduled(x, offs.to(dev), ex, pgu, pd, 0, 0, 0, sched, h, y2,
                                             fresh)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
        words = ws_[:256 + 4 * 1024].view(torch.int32).cpu()
        assert int(words[16]) == 0, "finished-CTA counter left set"
        assert int(words[64:64 + len(counts)].abs().sum()) == 0, "readiness counters left set"

    rng = np.random.default_rng(3)
    for sched in (None, moe.FfnSchedule(), moe.FfnSchedule(cta_pairs=1), moe.FfnSchedule(7, 0, 0, 0)):
        for n_seg in (1, 5, 40, 300):
            counts = [int(c) for c in rng.integers(0, 300, size=n_seg)]
            counts[0] = max(counts[0], 1)
            run(counts, sched if sched is not None else moe.FfnSchedule(), ws)
