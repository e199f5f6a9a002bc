"""The C-ABI library builds, loads without a GPU, exports every entry point
that include/moe.h declares, and rejects bad host-side arguments before any
CUDA call.  CPU only: no kernel is launched here."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from grouped_ffn_gb300 import build, moe
    build.build()
    return moe.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"moe_route", "moe_dispatch_layout", "moe_permute", "moe_grouped_ffn",
            "moe_combine", "moe_balance_stats"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert b"sm_103a" in lib.moe_version()


def test_status_strings(lib):
    from grouped_ffn_gb300 import moe
    for code, name in moe.STATUS_NAMES.items():
        s = moe.moe_status_string(code)
        assert s and s != "unknown status", name
    assert moe.moe_status_string(99) == "unknown status"


def test_workspace_size(lib):
    from grouped_ffn_gb300 import moe
    # status block (256) + FFN readiness counters (4096) + ticket block (256)
    # + one 32-bit flag per (1024-assignment tile, slot)
    assert moe.moe_workspace_size(4000, 2, 64) == 4608 + 8 * 64 * 4
    assert moe.moe_workspace_size(16384, 4, 40) == 4608 + 64 * 40 * 4
    assert moe.moe_workspace_size(0, 2, 64) == 4608 + 64 * 4
    assert moe.moe_workspace_size(-1, 2, 64) == 0


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


def test_host_validation_rejects_before_any_launch(lib):
    from grouped_ffn_gb300 import moe
    cfg = moe.RouteCfg(0, 2, 1, 1, 1)
    assert lib.moe_route(FAKE, -1, 64, ctypes.byref(cfg), FAKE, FAKE, None, 0, None) == 1
    assert lib.moe_route(FAKE, 8, 600, ctypes.byref(cfg), FAKE, FAKE, None, 0, None) == 2
    bad_k = moe.RouteCfg(0, 70, 1, 1, 1)
    assert lib.moe_route(FAKE, 8, 64, ctypes.byref(bad_k), FAKE, FAKE, None, 0, None) == 1
    grouped_softmax = moe.RouteCfg(0, 8, 8, 4, 2)
    assert lib.moe_route(FAKE, 8, 256, ctypes.byref(grouped_softmax), FAKE, FAKE, None, 0, None) == 2
    too_many_groups_kept = moe.RouteCfg(1, 8, 8, 9, 2)
    assert lib.moe_route(FAKE, 8, 256, ctypes.byref(too_many_groups_kept), FAKE, FAKE, None, 0, None) == 1
    assert lib.moe_route(None, 8, 64, ctypes.byref(cfg), FAKE, FAKE, None, 0, None) == 1
    # permute / combine: H must be a multiple of 8, workspace required
    assert lib.moe_permute(FAKE, 8, 12, 2, FAKE, FAKE, FAKE, 256, None) == 2
    assert lib.moe_permute(FAKE, 8, 256, 2, FAKE, FAKE, None, 0, None) == 6
    assert lib.moe_permute(ctypes.c_void_p(0x10008), 8, 256, 2, FAKE, FAKE, FAKE, 256, None) == 1
    assert lib.moe_combine(FAKE, FAKE, FAKE, 8, 17, 256, None, FAKE, FAKE, 256, None) == 2
    # grouped FFN: H % 256, I % 128, segment count limit
    args = lambda H, I, S: (FAKE, 16, FAKE, FAKE, S, 64, FAKE, FAKE, H, I, FAKE, FAKE, FAKE, 256, None)
    assert lib.moe_grouped_ffn(*args(300, 128, 64)) == 2
    assert lib.moe_grouped_ffn(*args(256, 96, 64)) == 2
    assert lib.moe_grouped_ffn(*args(256, 128, 2000)) == 2
    assert lib.moe_grouped_ffn(*args(256, 128, 0)) == 1
    # L2 weight prefetch: sizes and pointers first; T = 0 or a budget below one
    # 32 KiB k-block launches nothing
    pl = moe.PlacementC(64, 64, 8, 8, FAKE.value, FAKE.value, FAKE.value, FAKE.value, None)
    pf = lambda ids, T, H, nbytes: lib.moe_prefetch_ffn_weights(ids, T, 2, ctypes.byref(pl), FAKE,
                                                                 H, 128, nbytes, None)
    assert pf(FAKE, -1, 256, 1 << 20) == 1
    assert pf(FAKE, 8, 300, 1 << 20) == 2
    assert pf(None, 8, 256, 1 << 20) == 1
    assert pf(FAKE, 8, 256, 1000) == 0
    assert pf(FAKE, 0, 256, 1 << 20) == 0
    # watchdog self-test: 1 us <= limit <= 2 s, a workspace with its status block
    assert lib.moe_selftest_wait_timeout(FAKE, 256, 0, None, None) == 1
    assert lib.moe_selftest_wait_timeout(FAKE, 256, 2_000_001, None, None) == 1
    assert lib.moe_selftest_wait_timeout(None, 0, 1000, None, None) == 6
    assert lib.moe_selftest_wait_timeout(FAKE, 16, 1000, None, None) == 6
    # a tile list of 2^31 tiles or more: 2^24 m-blocks times (1024/128 + 30720/256) n-blocks
    assert lib.moe_grouped_ffn(FAKE, (1 << 31) - 1, FAKE, FAKE, 1, 1, FAKE, FAKE, 30720, 1024,
                               FAKE, FAKE, FAKE, 256, None) == 2
    # layout: slot limit, workspace size
    pl = moe.PlacementC(64, 2000, 8, 8, FAKE.value, FAKE.value, FAKE.value, FAKE.value, None)
    assert lib.moe_dispatch_layout(FAKE, 8, 2, ctypes.byref(pl), FAKE, FAKE, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, 1 << 20, None) == 2
    pl = moe.PlacementC(64, 64, 8, 8, FAKE.value, FAKE.value, FAKE.value, FAKE.value, None)
    assert lib.moe_dispatch_layout(FAKE, 8, 2, ctypes.byref(pl), FAKE, FAKE, FAKE, FAKE, FAKE,
                                   FAKE, FAKE, 256, None) == 6
    assert lib.moe_balance_stats(FAKE, 0, FAKE, FAKE, FAKE, None, 0, None) == 1
    # fixed-capacity layout: cap >= 1, S*cap < 2^31, workspace
    pl = moe.PlacementC(64, 64, 8, 8, FAKE.value, FAKE.value, FAKE.value, FAKE.value, None)
    lay = lambda cap, wsb: lib.moe_dispatch_layout_masked(
        FAKE, 8, 2, ctypes.byref(pl), cap, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsb, None)
    assert lay(0, 1 << 20) == 1
    assert lay(1 << 26, 1 << 20) == 2
    assert lay(4, 256) == 6
    # masked FFN: cap >= 1; masked permute / combine keep the plain checks
    assert lib.moe_grouped_ffn_masked(FAKE, 0, FAKE, FAKE, 4, 8, FAKE, FAKE, 256, 128, FAKE, FAKE,
                                      FAKE, 1 << 16, None) == 1
    assert lib.moe_grouped_ffn_masked(FAKE, 8, FAKE, FAKE, 4, 8, FAKE, FAKE, 300, 128, FAKE, FAKE,
                                      FAKE, 1 << 16, None) == 2
    assert lib.moe_permute_masked(FAKE, 8, 12, 2, FAKE, 16, FAKE, FAKE, 256, None) == 2
    assert lib.moe_permute_masked(FAKE, 8, 256, 2, FAKE, -1, FAKE, FAKE, 256, None) == 1
    assert lib.moe_combine_masked(FAKE, 16, FAKE, FAKE, 8, 17, 256, None, FAKE, FAKE, 256, None) == 2
    # FP8 dispatch: H % 128, alignment of the code buffer, masked geometry
    assert lib.moe_permute_fp8(FAKE, 8, 192, 2, FAKE, 16, FAKE, FAKE, FAKE, 256, None) == 2
    assert lib.moe_permute_fp8(FAKE, 8, 256, 2, FAKE, 16, ctypes.c_void_p(0x10004), FAKE, FAKE,
                               256, None) == 1
    assert lib.moe_permute_fp8(FAKE, 8, 256, 2, FAKE, 16, FAKE, FAKE, None, 0, None) == 6
    assert lib.moe_dequant_fp8(FAKE, FAKE, 10, 256, 3, FAKE, FAKE, None, 0, None) == 1
    assert lib.moe_dequant_fp8(FAKE, FAKE, 10, 200, 0, None, FAKE, None, 0, None) == 2


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from grouped_ffn_gb300 import moe
    with pytest.raises(TypeError):
        moe.moe_route(torch.zeros(4, 8), moe.RouteCfg(0, 2, 1, 1, 1),
                      torch.zeros(4, 2, dtype=torch.int32), torch.zeros(4, 2))
