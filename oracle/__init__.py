"""CPU oracle of the MoE-layer hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python
binding) never imports or calls it, and the two share no code: only the
seeded input generators in `workloads` feed both.

Each function is the plain definition of one step, written for a reader to
check against the pages by eye: fp64 arithmetic, library primitives
(sort, matmul, exp) as steps, no blocking or fusion.

Sources (page title, section):
  [MoE14]  "14. Serving Mixture-of-Experts Models" -- "Follow one token
           through an MoE layer" (router, the four runtime steps), "Price
           one dispatch", "The slowest expert sets the pace" (balancedness),
           "Worked example: balance the busiest rank",
           "The network topology is visible in every MoE layer" (replica
           preference).
  [MoEInf] "Mixture-of-Experts Inference: parallelism, communication, and
           load balancing" -- "MoE architecture recap" (grouped routing,
           shared experts), "Optimized kernels for MoE" (grouped GEMM,
           contiguous layout).
  [Zepp]   "Zepp: Accelerating Distributed MoE Serving under Relaxed Balance
           Constraints" -- Section 2 (top-k router, dispatch/combine),
           Section 4.1 (replicas, placement).

Readings where the pages are silent (each also listed in the design notes):
  * top-k order: descending score, ties to the lower expert id; selection
    compares the fp32 logits (softmax and sigmoid are monotone).
  * softmax weights are renormalised over the selected k.
  * group-limited routing: contiguous groups of E/n_groups experts; group
    score = fp64 sum of the fp64 sigmoids of the group's top-`group_topn`
    logits (taken in descending order); top `topk_groups` groups by
    (score desc, group id asc); weights = selected sigmoids / their sum.
  * expert FFN = SwiGLU: h = bf16(silu(x Wg^T) * (x Wu^T)), y = bf16(h Wd^T),
    silu(g) = g / (1 + e^-g); fp64 here.
  * combine: y[t] = bf16(shared[t] + sum_j w[t,j] * y_perm[dest_row[t,j]]).
  * balancedness: total / (R * max) in fp64, and 1.0 when nothing is routed.

Pins for every function live in tests/test_oracle_pins.py (brute force,
closed forms, the pages' worked examples); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------------ bf16
def bf16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (8 significant bits), ties to
    even, returning fp64.  Done in one step from fp64 so there is no double
    rounding through fp32.  (Finite inputs; magnitudes in the normal bf16
    range.)"""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> fp64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """fp64 values that are already bf16-representable -> uint16 patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------ route
def _order_desc_lower_id(scores_row: np.ndarray) -> np.ndarray:
    """Indices sorted by (score descending, index ascending)."""
    idx = np.arange(scores_row.shape[0])
    return np.lexsort((idx, -scores_row.astype(np.float64)))


def route_softmax_topk(logits: np.ndarray, k: int):
    """Softmax router with top-k ([MoE14] "Follow one token through an MoE
    layer": expert ids and weights per token; [Zepp] Section 2: a learned
    router selects the top-k experts).

    Returns (ids int32 [T,k], weights fp64 [T,k]).  The probabilities of the
    full softmax are renormalised over the k selected experts.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        row = logits[t]
        order = _order_desc_lower_id(row)[:k]
        l64 = row.astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        ids[t] = order
        w[t] = p[order] / p[order].sum()
    return ids, w


def sigmoid64(x) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def route_group_limited(logits: np.ndarray, k: int, n_groups: int,
                        topk_groups: int, group_topn: int):
    """Group-limited sigmoid router ([MoEInf] "MoE architecture recap": the
    routed experts are divided into groups; the router first picks a limited
    number of groups, then the top experts within them).

    Returns (ids int32 [T,k], weights fp64 [T,k], min relative group-score
    margin between the last kept and the first dropped group over all
    tokens, for near-tie reporting).
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    gs = E // n_groups
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    min_margin = np.inf
    for t in range(T):
        row = logits[t]
        gscore = np.empty(n_groups, dtype=np.float64)
        for g in range(n_groups):
            members = row[g * gs:(g + 1) * gs]
            top = _order_desc_lower_id(members)[:group_topn]
            s = 0.0
            for i in top:                       # descending order
                s = s + float(sigmoid64(members[i]))
            gscore[g] = s
        gorder = _order_desc_lower_id(gscore)
        kept = np.sort(gorder[:topk_groups])
        if topk_groups < n_groups:
            a, b = gscore[gorder[topk_groups - 1]], gscore[gorder[topk_groups]]
            min_margin = min(min_margin, (a - b) / max(abs(a), 1e-300))
        cand = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in kept])
        sub = _order_desc_lower_id(row[cand])[:k]
        chosen = cand[sub]
        s = sigmoid64(row[chosen])
        ids[t] = chosen
        w[t] = s / s.sum()
    return ids, w, min_margin


# ------------------------------------------------------------------ layout
def choose_slot(e: int, t: int, pl) -> int:
    """Physical slot that serves assignment (token t, expert e).

    One copy: its slot.  Several copies: the copy on token t's own node
    (the lowest such rank), else copy number (t mod n_copies) in ascending
    rank order.  This is the fixed replica rule of the replica workload;
    its preference order (same node first, else spread) follows [MoE14]
    "The network topology is visible in every MoE layer".
    """
    lo, hi = int(pl.rep_offsets[e]), int(pl.rep_offsets[e + 1])
    reps = [int(s) for s in pl.rep_slots[lo:hi]]
    if len(reps) == 1:
        return reps[0]
    src = int(pl.token_src_rank[t]) if pl.token_src_rank is not None else t % pl.n_ranks
    node = src // pl.ranks_per_node
    for s in reps:                                   # ascending rank
        if int(pl.slot_rank[s]) // pl.ranks_per_node == node:
            return s
    return reps[t % len(reps)]


def dispatch_layout(topk_ids: np.ndarray, pl) -> Dict[str, np.ndarray]:
    """Dispatch packing ([MoE14] "Follow one token", step 1: a permutation
    built from a histogram over the expert ids so that kernels see
    contiguous per-expert segments; here one segment per physical slot,
    ordered by (rank, expert), so each simulated rank's rows are contiguous
    as they would be after step 2's send to the owner rank).

    Assignment a = t*k + j.  Rows of a segment keep assignment order
    (stable).  Written as the literal definition: walk the assignments in
    order, append each to its slot's list, concatenate the lists.
    """
    T, k = topk_ids.shape
    A = T * k
    slot = np.array([choose_slot(int(topk_ids[a // k, a % k]), a // k, pl) for a in range(A)],
                    dtype=np.int32)
    return dispatch_layout_from_slots(topk_ids, slot, pl)


def dispatch_layout_from_slots(topk_ids: np.ndarray, slot: np.ndarray, pl) -> Dict[str, np.ndarray]:
    """The same packing when each assignment's slot is already chosen (for
    example by route_replicas_waterfill)."""
    T, k = topk_ids.shape
    S = pl.n_slots
    A = T * k
    slot = np.asarray(slot, dtype=np.int32)
    lists = [[] for _ in range(S)]
    for a in range(A):
        lists[int(slot[a])].append(a)
    seg_counts = np.array([len(l) for l in lists], dtype=np.int32)
    seg_offsets = np.zeros(S + 1, dtype=np.int32)
    seg_offsets[1:] = np.cumsum(seg_counts)
    src_assign = np.array([a for l in lists for a in l], dtype=np.int32)
    dest_row = np.empty(A, dtype=np.int32)
    dest_row[src_assign] = np.arange(A, dtype=np.int32)
    rank_counts = np.zeros(pl.n_ranks, dtype=np.int32)
    for s in range(S):
        rank_counts[int(pl.slot_rank[s])] += seg_counts[s]
    return dict(slot=slot, seg_counts=seg_counts, seg_offsets=seg_offsets,
                dest_row=dest_row, src_assign=src_assign, rank_counts=rank_counts)


def dispatch_layout_masked(topk_ids: np.ndarray, pl, cap: int,
                           slot: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Fixed-capacity ("masked") layout: every slot owns `cap` rows whatever
    its load, so the buffers and launches have the same shape every step
    ([MoEInf] "Communication pressure", prefill and decode kernel layouts:
    decode pads tokens into fixed-size masked layouts so that one captured
    CUDA graph can be replayed; [MoE14] "Capacity, padding, and the drop
    decision": a fixed per-expert capacity, and assignments beyond it are
    dropped, their output for the layer being zero).

    Slot s owns rows [s*cap, (s+1)*cap).  Walking the assignments in order,
    the first `cap` of slot s take rows s*cap, s*cap+1, ...; later ones are
    dropped (dest_row -1).  Returns slot, seg_counts (the demand, before
    dropping), masked_m (rows used: min(demand, cap)), dest_row,
    src_assign [S*cap] (-1 on unused rows), rank_counts (rows each rank
    executes: the sum of its slots' masked_m) and n_dropped."""
    T, k = topk_ids.shape
    S = pl.n_slots
    A = T * k
    if slot is None:
        slot = np.array([choose_slot(int(topk_ids[a // k, a % k]), a // k, pl) for a in range(A)],
                        dtype=np.int32)
    slot = np.asarray(slot, dtype=np.int32)
    seg_counts = np.zeros(S, dtype=np.int32)
    dest_row = np.full(A, -1, dtype=np.int32)
    src_assign = np.full(S * cap, -1, dtype=np.int32)
    for a in range(A):
        s = int(slot[a])
        pos = int(seg_counts[s])
        seg_counts[s] += 1
        if pos < cap:
            dest_row[a] = s * cap + pos
            src_assign[s * cap + pos] = a
    masked_m = np.minimum(seg_counts, cap).astype(np.int32)
    rank_counts = np.zeros(pl.n_ranks, dtype=np.int32)
    for s in range(S):
        rank_counts[int(pl.slot_rank[s])] += masked_m[s]
    n_dropped = int(seg_counts.sum() - masked_m.sum())
    return dict(slot=slot, seg_counts=seg_counts, masked_m=masked_m, dest_row=dest_row,
                src_assign=src_assign, rank_counts=rank_counts, n_dropped=n_dropped)


def grouped_ffn_masked(x_perm: np.ndarray, cap: int, masked_m: np.ndarray,
                       seg_expert: np.ndarray, w_gate_up, w_down, I: int):
    """The grouped FFN on a fixed-capacity layout: slot s runs expert
    seg_expert[s] on its rows [s*cap, s*cap + masked_m[s]); other rows are
    padding and come back as zero here.  Same per-row definition as
    grouped_ffn."""
    S = len(masked_m)
    H = x_perm.shape[1]
    h_out = np.zeros((S * cap, I))
    y_out = np.zeros((S * cap, H))
    for s in range(S):
        m = int(masked_m[s])
        if m == 0:
            continue
        r0 = s * cap
        e = int(seg_expert[s])
        h, y = swiglu_expert(x_perm[r0:r0 + m], np.asarray(w_gate_up[e], np.float64),
                             np.asarray(w_down[e], np.float64), I)
        h_out[r0:r0 + m] = h
        y_out[r0:r0 + m] = y
    return h_out, y_out


# ------------------------------------------------------------------ permute
def permute(x: np.ndarray, dest_row: np.ndarray, k: int,
            n_rows: Optional[int] = None) -> np.ndarray:
    """x_perm[dest_row[t*k+j]] = x[t] ([MoE14] "Price one dispatch": every
    assignment carries one copy of its token's hidden row).  Works on any
    dtype, so bf16 bit patterns are moved unchanged.  n_rows: rows of the
    output (default T*k); an assignment with dest_row -1 was dropped by a
    fixed-capacity layout and moves nothing.  Rows no assignment lands on
    are zero here (the GPU leaves them unwritten)."""
    T = x.shape[0]
    out = np.zeros((T * k if n_rows is None else n_rows,) + x.shape[1:], dtype=x.dtype)
    for a in range(T * k):
        if dest_row[a] >= 0:
            out[dest_row[a]] = x[a // k]
    return out


# ------------------------------------------------------------------ FP8 dispatch
# [MoEInf] "Communication pressure": token activations can be quantized, for
# example to FP8, before dispatch, to shrink what the all-to-all moves.
# Readings: OCP FP8 E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3
# mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448);
# one scale per (token, 128 consecutive channels); the scale is the power of
# two 2^e with the smallest e such that the block's largest magnitude is at
# most 448 * 2^e (so x / 2^e is exact and only the rounding to E4M3 loses
# information), e clamped to [-126, 127], and e = 0 for an all-zero block;
# codes are x / 2^e rounded to the nearest E4M3 value, ties to the even
# code.  The receiver restores bf16(code_value * 2^e).
FP8_BLOCK = 128
E4M3_MAX = 448.0


def e4m3_value(code) -> np.ndarray:
    """E4M3 codes (uint8) -> fp64 values, from the bit fields: exponent
    field 0 is subnormal (m/8 * 2^-6), otherwise (1 + m/8) * 2^(E-7); the
    two NaN codes map to nan."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(E == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(E.astype(np.float64) - 7))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


_E4M3_POS = e4m3_value(np.arange(0x7F))   # the 127 finite non-negative values, ascending


def e4m3_encode(v) -> np.ndarray:
    """fp64 values with |v| <= 448 -> the E4M3 code of the nearest value,
    ties to the even code (the one whose lowest mantissa bit is 0).  Found
    by search in the table of all finite values, so no bit trick is
    involved.  The sign bit is kept for zero results (-0 -> 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    if np.any(a > E4M3_MAX) or np.any(np.isnan(v)):
        raise ValueError("e4m3_encode: value outside [-448, 448]")
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def fp8_block_exponent(amax: float) -> int:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-126, 127];
    0 when amax is 0.  Exact: candidates are checked with exact power-of-two
    scaling (ldexp) in fp64."""
    amax = float(amax)
    if amax == 0.0:
        return 0
    e = int(np.ceil(np.log2(amax / E4M3_MAX)))
    while amax > np.ldexp(E4M3_MAX, e):
        e += 1
    while amax <= np.ldexp(E4M3_MAX, e - 1):
        e -= 1
    return int(min(max(e, -126), 127))


def quantize_fp8_blocks(x_bits: np.ndarray):
    """bf16 rows (uint16 [T, H], H a multiple of 128) -> (codes uint8 [T, H],
    scales fp32 [T, H/128] holding 2^e).  Per block: e from the largest
    magnitude, codes = e4m3_encode(x / 2^e)."""
    x = bf16_bits_to_f64(x_bits)
    T, H = x.shape
    nb = H // FP8_BLOCK
    codes = np.empty((T, H), dtype=np.uint8)
    scales = np.empty((T, nb), dtype=np.float32)
    for t in range(T):
        for b in range(nb):
            blk = x[t, b * FP8_BLOCK:(b + 1) * FP8_BLOCK]
            e = fp8_block_exponent(np.max(np.abs(blk)))
            codes[t, b * FP8_BLOCK:(b + 1) * FP8_BLOCK] = e4m3_encode(np.ldexp(blk, -e))
            scales[t, b] = np.float32(np.ldexp(1.0, e))
    return codes, scales


def dequantize_fp8_blocks(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """(codes [n, H], scales [n, H/128]) -> bf16 bit patterns [n, H] of
    bf16(code_value * scale), rounded to nearest, ties to even."""
    vals = e4m3_value(codes) * np.repeat(np.asarray(scales, np.float64), FP8_BLOCK, axis=1)
    # below 2^-126 bf16 is subnormal: a fixed step of 2^-133, ties to even
    tiny = np.abs(vals) < 2.0 ** -126
    rounded = np.where(tiny, np.ldexp(np.rint(np.ldexp(vals, 133)), -133),
                       bf16_round(np.where(tiny, 1.0, vals)))
    return f64_to_bf16_bits(rounded)


# ------------------------------------------------------------------ expert FFN
def silu64(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_expert(x_rows: np.ndarray, w_gate_up_e: np.ndarray,
                  w_down_e: np.ndarray, I: int):
    """One expert's gated MLP on a block of rows, fp64 from bf16 values.

    x_rows [n,H], w_gate_up_e [2I,H] (gate rows then up rows), w_down_e [H,I],
    all fp64 holding bf16 values.  Returns (h, y) with h rounded to bf16
    before the down projection and y rounded to bf16.
    """
    g = x_rows @ w_gate_up_e[:I].T
    u = x_rows @ w_gate_up_e[I:].T
    h = bf16_round(silu64(g) * u)
    y = bf16_round(h @ w_down_e.T)
    return h, y


def grouped_ffn(x_perm: np.ndarray, seg_offsets: np.ndarray, seg_expert: np.ndarray,
                w_gate_up: np.ndarray, w_down: np.ndarray, I: int,
                rows: Optional[np.ndarray] = None):
    """Grouped expert FFN ([MoE14] "Follow one token", step 3: one kernel
    runs every expert's segment as a matrix with its own row count;
    [MoEInf] "Optimized kernels for MoE": grouped GEMM, contiguous layout).

    Segment s covers rows [seg_offsets[s], seg_offsets[s+1]) and uses expert
    seg_expert[s].  Inputs are fp64 arrays of bf16 values; w_gate_up may be
    indexed lazily (any object with __getitem__ returning [2I,H]).
    rows: optional sorted subset of row indices to evaluate.  Returns
    (h [n,I], y [n,H]) for all rows or for `rows` in that order.
    """
    n_rows = x_perm.shape[0] if rows is None else len(rows)
    H = x_perm.shape[1]
    want = np.arange(x_perm.shape[0]) if rows is None else np.asarray(rows)
    h_out = np.zeros((n_rows, I))
    y_out = np.zeros((n_rows, H))
    seg_of = np.searchsorted(np.asarray(seg_offsets), want, side="right") - 1
    for s in np.unique(seg_of):
        sel = np.nonzero(seg_of == s)[0]
        e = int(seg_expert[s])
        h, y = swiglu_expert(x_perm[want[sel]], np.asarray(w_gate_up[e], np.float64),
                             np.asarray(w_down[e], np.float64), I)
        h_out[sel] = h
        y_out[sel] = y
    return h_out, y_out


# ------------------------------------------------------------------ combine
def combine_f64(y_perm: np.ndarray, dest_row: np.ndarray, topk_w: np.ndarray,
                shared: Optional[np.ndarray] = None, tokens=None) -> np.ndarray:
    """Inverse permutation followed by the router-weighted sum ([MoE14]
    "Follow one token", step 4; [Zepp] Section 2: outputs aggregated at each
    token's source), plus the shared expert's output with weight one
    ([MoEInf] "MoE architecture recap": shared experts see every token).
    fp64 accumulation, bf16 result.  tokens: optional subset.  An
    assignment dropped by a fixed-capacity layout (dest_row -1) adds
    nothing ([MoE14] "Capacity, padding, and the drop decision": a dropped
    token's output for the layer is zero)."""
    T, k = topk_w.shape
    ts = np.arange(T) if tokens is None else np.asarray(tokens)
    out = np.zeros((len(ts), y_perm.shape[1]))
    for i, t in enumerate(ts):
        acc = np.zeros(y_perm.shape[1]) if shared is None else shared[t].astype(np.float64)
        for j in range(k):
            if dest_row[t * k + j] < 0:      # dropped: its output is zero
                continue
            acc = acc + float(topk_w[t, j]) * y_perm[dest_row[t * k + j]]
        out[i] = bf16_round(acc)
    return out


_fma_lib = None


def build_c(force: bool = False) -> str:
    """Compile the oracle's C part (gcc, no CUDA) next to its source."""
    src = os.path.join(_HERE, "fma_combine.c")
    so = os.path.join(_HERE, "liboracle_fma.so")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", so, src, "-lm"])
    return so


def _fma():
    global _fma_lib
    if _fma_lib is None:
        lib = ctypes.CDLL(build_c())
        lib.oracle_combine_fma32.restype = None
        lib.oracle_combine_fma32.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        _fma_lib = lib
    return _fma_lib


def combine_fma32(y_perm_bits: np.ndarray, dest_row: np.ndarray, topk_w32: np.ndarray,
                  shared_bits: Optional[np.ndarray] = None) -> np.ndarray:
    """The combine with its fp32 evaluation order written out: per element,
    acc = shared (or 0); for j = 0..k-1: acc = fmaf(w[t,j], y, acc); result
    bf16 (nearest, ties to even).  Inputs/outputs are bf16 bit patterns
    (uint16).  This fixes one valid rounding order so that a stage fed the
    same y_perm can be compared bit for bit.  Terms with dest_row -1
    (dropped assignments) are skipped."""
    T, k = topk_w32.shape
    H = y_perm_bits.shape[1]
    yp = np.ascontiguousarray(y_perm_bits, dtype=np.uint16)
    dr = np.ascontiguousarray(dest_row, dtype=np.int32)
    w = np.ascontiguousarray(topk_w32, dtype=np.float32)
    sh = None if shared_bits is None else np.ascontiguousarray(shared_bits, dtype=np.uint16)
    out = np.empty((T, H), dtype=np.uint16)
    _fma().oracle_combine_fma32(yp.ctypes.data, dr.ctypes.data, w.ctypes.data,
                                None if sh is None else sh.ctypes.data,
                                T, k, H, out.ctypes.data)
    return out


# ------------------------------------------------------------------ balance
def balance_stats(rank_counts: np.ndarray):
    """Balancedness = mean per-rank load / busiest rank's load ([MoE14] "The
    slowest expert sets the pace": avg_tokens / max_tokens, 1.0 when
    perfectly balanced).  Loads count assignments, not unique tokens
    ([MoE14] "Price one dispatch").  Returns (balancedness, max, total)."""
    rc = np.asarray(rank_counts, dtype=np.int64)
    total = int(rc.sum())
    mx = int(rc.max()) if rc.size else 0
    if total == 0:
        return 1.0, mx, total
    return float(total) / (float(len(rc)) * float(mx)), mx, total


def balance_stats_layers(rank_counts: np.ndarray):
    """Balancedness of a step over several MoE layers ([MoE14] "The slowest
    expert sets the pace": avg_tokens / max_tokens, "summed across
    layers").  Reading: avg_tokens and max_tokens are each summed over the
    layers -- the sum of every layer's mean per-rank load over the sum of
    every layer's busiest-rank load; one layer gives balance_stats.
    rank_counts [L, R].  Returns (balancedness, sum of per-layer maxima,
    total); balancedness is 1.0 when nothing is routed."""
    rc = np.asarray(rank_counts, dtype=np.int64)
    L, R = rc.shape
    avg_sum = sum(float(rc[l].sum()) / float(R) for l in range(L))
    max_sum = int(sum(int(rc[l].max()) for l in range(L))) if R else 0
    total = int(rc.sum())
    if total == 0:
        return 1.0, max_sum, total
    return avg_sum / float(max_sum), max_sum, total


# ------------------------------------------------------------------ layer
def moe_layer_tokens(tokens, logits, x_bits, w_gate_up, w_down, pl, route_cfg,
                     shared_w=None, I=None, shared_I=None):
    """Whole layer for a subset of tokens, evaluated one token at a time from
    its definition: route the token, run each selected expert's FFN on its
    row, add the shared expert, weighted sum.  Replica choice does not change
    the value (copies hold identical weights), so it is not needed here.

    tokens: token indices; logits fp32 [T,E]; x_bits uint16 [T,H];
    w_gate_up / w_down: indexable by expert -> bf16 bit arrays;
    route_cfg: dict(score_fn, k, n_groups, topk_groups, group_topn).
    Returns y fp64 (bf16 values) [len(tokens), H].
    """
    tokens = np.asarray(tokens)
    lg = np.asarray(logits)[tokens]
    if route_cfg["score_fn"] == 0:
        ids, w = route_softmax_topk(lg, route_cfg["k"])
    else:
        ids, w, _ = route_group_limited(lg, route_cfg["k"], route_cfg["n_groups"],
                                        route_cfg["topk_groups"], route_cfg["group_topn"])
    w32 = w.astype(np.float32).astype(np.float64)   # the router emits fp32 weights
    out = np.zeros((len(tokens), x_bits.shape[1]))
    for i, t in enumerate(tokens):
        xr = bf16_bits_to_f64(x_bits[t])[None, :]
        acc = np.zeros(x_bits.shape[1])
        if shared_w is not None:
            _, ys = swiglu_expert(xr, bf16_bits_to_f64(shared_w[0]), bf16_bits_to_f64(shared_w[1]),
                                  shared_I)
            acc = acc + ys[0]
        for j in range(ids.shape[1]):
            e = int(ids[i, j])
            _, ye = swiglu_expert(xr, bf16_bits_to_f64(w_gate_up[e]), bf16_bits_to_f64(w_down[e]), I)
            acc = acc + w32[i, j] * ye[0]
        out[i] = bf16_round(acc)
    return out


# ------------------------------------------------------------------ replica routing
def replica_bounds(D: int, n: int, c_num: int, c_den: int):
    """Integer load targets and bounds for one expert's n replicas.

    [Zepp] Section 4.1 (Eq. 1): q_j is the expert's total demand divided
    evenly over its replicas, and each replica's load must stay within
    C * q_j of it; Section 5 rounds these to integers.  Reading: the
    integer even split q_p = floor(D/n) + (p < D mod n), slack
    floor(C * D / n) with C = c_num / c_den, bounds q_p -+ slack (lower
    bound at least 0).  sum(lo) <= D <= sum(hi) always holds."""
    base, rem = divmod(D, n)
    q = [base + (1 if p < rem else 0) for p in range(n)]
    slack = (c_num * D) // (c_den * n)
    lo = [max(0, qp - slack) for qp in q]
    hi = [qp + slack for qp in q]
    return q, lo, hi


def waterfill_expert(demand, rep_ranks, ranks_per_node, c_num, c_den):
    """Greedy water-filling of one expert's demand over its replicas.

    [Zepp] Section 5, "Routing": replicas on the source GPU are considered
    first, then other GPUs of the same node, then remote nodes; each
    allocation is limited by the receiving replica's remaining capacity
    while reserving enough unassigned demand for the other replicas' lower
    bounds.  Sources are taken in ascending rank, replicas in ascending
    rank within each pass.  A fourth pass places any demand the reserve
    rule held back: first into replicas still below their lower bound, then
    into any replica with capacity (this always completes: see the design
    notes).

    demand: dict rank -> count; rep_ranks: ascending ranks of the replicas.
    Returns (allocations, loads, lo, hi) with allocations a dict
    rank -> list of (replica position, count) in the order made.
    """
    n = len(rep_ranks)
    D = sum(demand.values())
    _, lo, hi = replica_bounds(D, n, c_num, c_den)
    load = [0] * n
    left = dict(demand)
    alloc = {i: [] for i in demand}
    U = D
    node = lambda r: r // ranks_per_node

    def give(i, p, x):
        nonlocal U
        if x <= 0:
            return
        left[i] -= x
        load[p] += x
        U -= x
        alloc[i].append((p, x))

    def allow(p):
        others = sum(max(0, lo[q] - load[q]) for q in range(n) if q != p)
        return max(0, min(hi[p] - load[p], U - others))

    sources = sorted(demand)
    passes = [lambda i, r: r == i,
              lambda i, r: r != i and node(r) == node(i),
              lambda i, r: node(r) != node(i)]
    for in_pass in passes:
        for i in sources:
            for p in range(n):
                if left[i] > 0 and in_pass(i, rep_ranks[p]):
                    give(i, p, min(left[i], allow(p)))
    for i in sources:
        for p in range(n):
            if left[i] > 0 and lo[p] - load[p] > 0:
                give(i, p, min(left[i], lo[p] - load[p]))
        for p in range(n):
            if left[i] > 0:
                give(i, p, min(left[i], hi[p] - load[p]))
    assert U == 0
    return alloc, load, lo, hi


def locality_order(i: int, rep_ranks, ranks_per_node: int):
    """Replica positions in the order source rank i prefers them: its own
    GPU, then its node (ascending rank), then remote (ascending rank)."""
    node = lambda r: r // ranks_per_node
    n = len(rep_ranks)
    return ([p for p in range(n) if rep_ranks[p] == i] +
            [p for p in range(n) if rep_ranks[p] != i and node(rep_ranks[p]) == node(i)] +
            [p for p in range(n) if node(rep_ranks[p]) != node(i)])


def route_replicas_waterfill(topk_ids: np.ndarray, pl, c_num: int, c_den: int):
    """Locality-preferred choice of the replica serving each assignment
    ([Zepp] Section 4.1 "Locality-preferred token routing" and Section 5).

    Per expert with several replicas: demand d_i = assignments of that
    expert whose token lives on rank i; the water-filling above fixes how
    many of rank i's assignments each replica serves (M[i][p]); rank i's
    assignments, in ascending order, then fill those destinations in its
    locality order (own GPU, own node, remote; ascending rank within each).  Experts
    with one replica keep it.  Returns (slot [A] int32, inter_node count)."""
    T, k = topk_ids.shape
    A = T * k
    ids = topk_ids.reshape(-1)
    src = np.array([int(pl.token_src_rank[a // k]) if pl.token_src_rank is not None
                    else (a // k) % pl.n_ranks for a in range(A)])
    slot = np.empty(A, dtype=np.int32)
    for e in range(pl.n_experts):
        reps = [int(s) for s in pl.rep_slots[pl.rep_offsets[e]:pl.rep_offsets[e + 1]]]
        mine = np.nonzero(ids == e)[0]
        if len(reps) == 1:
            slot[mine] = reps[0]
            continue
        rep_ranks = [int(pl.slot_rank[s]) for s in reps]
        demand = {}
        for a in mine:
            demand[int(src[a])] = demand.get(int(src[a]), 0) + 1
        alloc, _, _, _ = waterfill_expert(demand, rep_ranks, pl.ranks_per_node, c_num, c_den)
        for i, lst in alloc.items():
            count = [0] * len(reps)                          # M[i][p]
            for p, x in lst:
                count[p] += x
            rows = [a for a in mine if src[a] == i]          # ascending assignment order
            pos = 0
            for p in locality_order(i, rep_ranks, pl.ranks_per_node):
                slot[rows[pos:pos + count[p]]] = reps[p]
                pos += count[p]
    node_of = lambda r: r // pl.ranks_per_node
    inter = int(sum(node_of(int(pl.slot_rank[slot[a]])) != node_of(int(src[a])) for a in range(A)))
    return slot, inter


def refine_consolidate(topk_ids: np.ndarray, slot: np.ndarray, pl):
    """Greedy refinement of a feasible replica routing ([Zepp] Section 5,
    "Routing": starting from the water-filling's assignments, consolidate
    each token's remote expert requests onto fewer nodes while keeping the
    same load bounds; Section 1: remaining requests go to fewer remote
    nodes).

    Readings:
      * The water-filling's counts M[i][p] (assignments of source rank i
        served by replica p) stay fixed, so every replica's load, every
        source's row total, the bounds of Eq. 1 and the number of
        inter-node assignments are unchanged; only which of a source's
        remote assignments takes which remote replica changes.
      * Assignments that the water-filling served on the source's own node
        keep their slot (its fill order gives the node-local copies to a
        source's earliest assignments, and the refinement keeps that), as do
        assignments of experts with one copy.
      * Sources are independent (they share no counts).  Within source
        rank i, tokens go in ascending order; each token's re-choosable
        requests (replicated expert, remote copy) are covered greedily by
        nodes: first a node the token already sends to (a fixed remote
        request or an earlier choice), then the node covering the most of
        its open requests, ties to the lower node id; a request takes the
        lowest-rank copy of its expert on that node that still has count
        left for source i.
      * A source keeps its refined choices only if they do not raise its
        number of distinct (token, remote node) pairs (the merged dispatch
        messages of [Zepp] Section 4.2); otherwise its original ones.

    Returns (slot [A] int32, pairs before, pairs after)."""
    T, k = topk_ids.shape
    A = T * k
    ids = topk_ids.reshape(-1)
    slot = np.asarray(slot, dtype=np.int32)
    out = slot.copy()
    rpn = pl.ranks_per_node
    node_of = lambda r: int(r) // rpn
    src_of = [int(pl.token_src_rank[t]) if pl.token_src_rank is not None else t % pl.n_ranks
              for t in range(T)]
    reps_of = [[int(s) for s in pl.rep_slots[pl.rep_offsets[e]:pl.rep_offsets[e + 1]]]
               for e in range(pl.n_experts)]

    def pairs(t, sl):
        n_t = node_of(src_of[t])
        return len({node_of(pl.slot_rank[sl[t * k + j]]) for j in range(k)} - {n_t})

    before = after = 0
    for i in range(pl.n_ranks):
        toks = [t for t in range(T) if src_of[t] == i]
        n_i = node_of(i)
        # remaining count of source i's assignments per remote copy (slot)
        left = {}
        for t in toks:
            for j in range(k):
                a = t * k + j
                e = int(ids[a])
                s = int(slot[a])
                if len(reps_of[e]) > 1 and node_of(pl.slot_rank[s]) != n_i:
                    left[s] = left.get(s, 0) + 1
        cand = slot.copy()
        for t in toks:
            used = set()
            open_j = []
            for j in range(k):
                a = t * k + j
                e = int(ids[a])
                m = node_of(pl.slot_rank[int(slot[a])])
                if m == n_i:
                    continue
                if len(reps_of[e]) > 1:
                    open_j.append(j)
                else:
                    used.add(m)
            while open_j:
                cover = {}
                for j in open_j:
                    e = int(ids[t * k + j])
                    for m in {node_of(pl.slot_rank[s]) for s in reps_of[e]
                              if left.get(s, 0) > 0 and node_of(pl.slot_rank[s]) != n_i}:
                        cover.setdefault(m, []).append(j)
                best = min(cover, key=lambda m: (m not in used, -len(cover[m]), m))
                taken = []
                for j in cover[best]:
                    e = int(ids[t * k + j])
                    on_best = [s for s in reps_of[e]
                               if left.get(s, 0) > 0 and node_of(pl.slot_rank[s]) == best]
                    if not on_best:      # only when a token repeats an expert id
                        continue
                    s = min(on_best, key=lambda s: int(pl.slot_rank[s]))
                    left[s] -= 1
                    cand[t * k + j] = s
                    taken.append(j)
                used.add(best)
                open_j = [j for j in open_j if j not in taken]
        b = sum(pairs(t, slot) for t in toks)
        c = sum(pairs(t, cand) for t in toks)
        before += b
        if c <= b:
            for t in toks:
                out[t * k:(t + 1) * k] = cand[t * k:(t + 1) * k]
            after += c
        else:
            after += b
    return out, before, after


# ------------------------------------------------------------------ merge (simulated)
def dispatch_messages(slot: np.ndarray, pl, T: int, k: int):
    """Inter-node dispatch transfers of one step, before and after merge
    ([Zepp] Section 3.2 "Redundant Tokens" and Section 4.2 "Merge": a token
    whose experts share a remote node crosses the network once).  Returns
    (remote assignments, unique (token, remote node) pairs)."""
    before, pairs = 0, set()
    for a in range(T * k):
        t = a // k
        src = int(pl.token_src_rank[t]) if pl.token_src_rank is not None else t % pl.n_ranks
        dn = int(pl.slot_rank[int(slot[a])]) // pl.ranks_per_node
        if dn != src // pl.ranks_per_node:
            before += 1
            pairs.add((t, dn))
    return before, len(pairs)


def combine_merged_fma32(y_perm_bits, dest_row, topk_w32, node, shared_bits=None):
    """Combine with node-local pre-reduction; see oracle_combine_merged_fma32
    in fma_combine.c for the order of operations.  bf16 bit patterns in and
    out; node[a] is assignment a's destination node."""
    T, k = topk_w32.shape
    H = y_perm_bits.shape[1]
    yp = np.ascontiguousarray(y_perm_bits, dtype=np.uint16)
    dr = np.ascontiguousarray(dest_row, dtype=np.int32)
    w = np.ascontiguousarray(topk_w32, dtype=np.float32)
    nd = np.ascontiguousarray(node, dtype=np.int32)
    sh = None if shared_bits is None else np.ascontiguousarray(shared_bits, dtype=np.uint16)
    out = np.empty((T, H), dtype=np.uint16)
    lib = _fma()
    if not hasattr(lib, "_merged_ready"):
        lib.oracle_combine_merged_fma32.restype = None
        lib.oracle_combine_merged_fma32.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        lib._merged_ready = True
    lib.oracle_combine_merged_fma32(yp.ctypes.data, dr.ctypes.data, w.ctypes.data, nd.ctypes.data,
                                    None if sh is None else sh.ctypes.data, T, k, H,
                                    out.ctypes.data)
    return out


def combine_merged_f64(y_perm, dest_row, topk_w, node, shared=None):
    """The same pre-reduction in fp64 with the bf16 rounding of each node's
    partial sum kept (it is the transferred payload); bf16 result."""
    T, k = topk_w.shape
    out = np.zeros((T, y_perm.shape[1]))
    for t in range(T):
        acc = np.zeros(y_perm.shape[1]) if shared is None else shared[t].astype(np.float64)
        for n in sorted(set(int(v) for v in node[t * k:(t + 1) * k])):
            part = np.zeros(y_perm.shape[1])
            for j in range(k):
                if int(node[t * k + j]) == n:
                    part = part + float(topk_w[t, j]) * y_perm[dest_row[t * k + j]]
            acc = acc + bf16_round(part)
        out[t] = bf16_round(acc)
    return out
