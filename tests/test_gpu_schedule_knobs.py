"""The grouped FFN's schedule switches change how tiles are run, never the
arithmetic of a row: the layer's h, y_perm and y are bit-identical under
every setting.  MOE_FFN_PH1_SHIFT (phase-1 positions given first to the CTAs
with one gate/up tile fewer) and MOE_FFN_INTERLEAVE=0 (plain segment order)
change which CTA runs a tile and when; MOE_FFN_SMALL_TILES=0 runs segments
of at most 64 rows as 128-row tiles instead of M = 64 ones.  The switches are
read once per process, so each setting runs the same seeded layer in a child
process, which prints a hash of its outputs."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# 4000 tokens, top-2 over 64 experts with Zipf 1.0 skew and a shared expert
# in the routed launch: over 100 m-blocks, so the gate/up phase has more
# tiles than the 152 CTAs and a partial last wave that the shift rebalances,
# and the skew's tail has many segments of at most 64 rows.
CHILD = r"""
import hashlib, sys
import torch
sys.path.insert(0, sys.argv[1])
import workloads as wl
from grouped_ffn_gb300 import MoELayer, moe

dev = torch.device("cuda", 0)
w = wl.Workload("schedule", 91, T=4000, H=1024, E=64, k=2, I=512, R=8, ranks_per_node=8,
                shared_I=512, zipf_s=1.0)
pl = wl.make_placement(w)
logits, x = wl.make_logits(w, dev), wl.make_x(w, dev)
sgu, sd = wl.make_shared_weights(w, dev)
layer = MoELayer(H=w.H, I=w.I, E=w.E, k=w.k, placement=moe.DevicePlacement.from_tables(pl, dev),
                 w_gate_up=wl.make_w_gate_up(w, dev), w_down=wl.make_w_down(w, dev),
                 max_tokens=w.T, shared_w_gate_up=sgu, shared_w_down=sd, device=dev)
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
print("SMALL", small)
print("HASH", h.hexdigest())
"""


KNOBS = ("MOE_FFN_PH1_SHIFT", "MOE_FFN_INTERLEAVE", "MOE_FFN_SMALL_TILES")


def _run(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in KNOBS}
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("HASH ")]
    small = [ln for ln in r.stdout.splitlines() if ln.startswith("SMALL ")]
    assert len(lines) == 1 and len(small) == 1, r.stdout[-2000:]
    return lines[0].split()[1], int(small[0].split()[1])


def test_tile_schedules_give_identical_bits():
    from grouped_ffn_gb300 import build
    build.build()
    ref, small = _run({})
    assert small >= 8, small   # the M = 64 path is exercised
    for extra in ({"MOE_FFN_PH1_SHIFT": "0"}, {"MOE_FFN_PH1_SHIFT": "7"},
                  {"MOE_FFN_INTERLEAVE": "0"},
                  {"MOE_FFN_INTERLEAVE": "0", "MOE_FFN_PH1_SHIFT": "0"},
                  {"MOE_FFN_SMALL_TILES": "0"},
                  {"MOE_FFN_SMALL_TILES": "0", "MOE_FFN_INTERLEAVE": "0"}):
        assert _run(extra) == (ref, small), extra
