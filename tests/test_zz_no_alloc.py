"""moe_dispatch_layout_noalloc, the layout entry point for callers that
cannot allocate device memory (for instance a serving engine whose free HBM
is all promised to its weight and KV-cache pools, or a plugin run by another
runtime that gives it no workspace and no cudaMalloc).  It must give exactly
the results of moe_dispatch_layout, call after call, while its scratch lives
in the library's fixed device array.  This file is collected last so that a
stop-at-first-failure run has already run every other test."""

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from grouped_ffn_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _outputs(T, k, pl_dev):
    A = T * k
    mk = lambda n: torch.full((n,), -5, dtype=torch.int32, device="cuda")
    return [mk(A), mk(pl_dev.n_slots), mk(pl_dev.n_slots + 1), mk(A), mk(A), mk(pl_dev.n_ranks)]


def _ids(name, seed):
    w = wl.WORKLOADS[name]
    g = torch.Generator(device="cuda").manual_seed(seed)
    # random expert ids, distinct within a token
    scores = torch.rand(w.T, w.E, generator=g, device="cuda")
    ids = scores.topk(w.k, dim=1).indices.to(torch.int32).contiguous()
    return w, ids


@pytest.mark.parametrize("first,second", [("replica", "prefill"), ("group_limited", "tiny")])
def test_noalloc_layout_matches_workspace_layout_on_consecutive_calls(first, second):
    from grouped_ffn_gb300 import moe
    for i, name in enumerate([first, second, first]):
        w, ids = _ids(name, 100 + i)
        pl_dev = moe.DevicePlacement.from_tables(wl.make_placement(w))
        ws = moe.new_workspace(w.T, w.k, pl_dev.n_slots)
        ref = _outputs(w.T, w.k, pl_dev)
        moe.moe_dispatch_layout(ids, pl_dev, *ref, ws)
        got = _outputs(w.T, w.k, pl_dev)
        status = torch.zeros(3, dtype=torch.int32, device="cuda")
        moe.moe_dispatch_layout_noalloc(ids, pl_dev, *got, status=status)
        torch.cuda.synchronize()
        moe.moe_check_device_status(ws)
        assert status.tolist() == [0, 0, 0]
        for r, g in zip(ref, got):
            assert torch.equal(r, g), name


@pytest.mark.parametrize("name", ["prefill", "replica"])
def test_layout_after_an_empty_call_on_the_same_scratch(name):
    """A call with no assignments leaves the ticket and the look-back flags
    clear (its single scan CTA finalizes and writes no flag), so a following
    multi-tile call on the same scratch -- the library's fixed array, or a
    workspace -- still gives the workspace layout of a fresh workspace."""
    from grouped_ffn_gb300 import moe
    w, ids = _ids(name, 7)
    pl_dev = moe.DevicePlacement.from_tables(wl.make_placement(w))
    fresh = moe.new_workspace(w.T, w.k, pl_dev.n_slots)
    ref = _outputs(w.T, w.k, pl_dev)
    moe.moe_dispatch_layout(ids, pl_dev, *ref, fresh)
    # the library's scratch
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_layout_noalloc(ids[:0], pl_dev, *_outputs(0, w.k, pl_dev), status=status)
    got = _outputs(w.T, w.k, pl_dev)
    moe.moe_dispatch_layout_noalloc(ids, pl_dev, *got, status=status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0]
    for r, g in zip(ref, got):
        assert torch.equal(r, g), name
    # a workspace
    ws = moe.new_workspace(w.T, w.k, pl_dev.n_slots)
    moe.moe_dispatch_layout(ids[:0], pl_dev, *_outputs(0, w.k, pl_dev), ws)
    got = _outputs(w.T, w.k, pl_dev)
    moe.moe_dispatch_layout(ids, pl_dev, *got, ws)
    moe.moe_check_device_status(ws)
    for r, g in zip(ref, got):
        assert torch.equal(r, g), name


def test_noalloc_layout_rejects_requests_beyond_its_scratch():
    from grouped_ffn_gb300 import moe
    # 1024 slots x 1024 tiles of 1024 assignments needs more than 262144 flag words
    E = R = 1024
    pl = wl.placement_from_hosts(E, R, 8, wl.round_robin_hosts(E, R))
    pl_dev = moe.DevicePlacement.from_tables(pl)
    T, k = 4096 * 256 // 2, 2
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    out = _outputs(T, k, pl_dev)
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_layout_noalloc(ids, pl_dev, *out, status=status)
    assert ei.value.status == 2          # MOE_ERR_UNSUPPORTED, nothing launched


def test_noalloc_device_error_reaches_status_and_the_next_call_is_clean():
    """An expert id out of range in a layout of several 1024-assignment tiles
    is reported in the caller's status array (MOE_ERR_DEVICE_INDEX) rather
    than dropped; the shared scratch it leaves behind does not disturb the
    next call, which again gives the workspace layout."""
    from grouped_ffn_gb300 import moe
    w, ids = _ids("prefill", 31)          # 8000 assignments: 2 tiles
    pl_dev = moe.DevicePlacement.from_tables(wl.make_placement(w))
    bad = ids.clone()
    bad[5000 // w.k, 0] = w.E + 3         # in the second tile
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_layout_noalloc(bad, pl_dev, *_outputs(w.T, w.k, pl_dev), status=status)
    torch.cuda.synchronize()
    assert status[0].item() == 4         # MOE_ERR_DEVICE_INDEX
    ws = moe.new_workspace(w.T, w.k, pl_dev.n_slots)
    ref = _outputs(w.T, w.k, pl_dev)
    moe.moe_dispatch_layout(ids, pl_dev, *ref, ws)
    moe.moe_check_device_status(ws)
    got = _outputs(w.T, w.k, pl_dev)
    status.zero_()
    moe.moe_dispatch_layout_noalloc(ids, pl_dev, *got, status=status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0]
    for r, g in zip(ref, got):
        assert torch.equal(r, g)
