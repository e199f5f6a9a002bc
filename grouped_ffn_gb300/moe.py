"""ctypes binding of libmoe.so (declared in include/moe.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Functions carry the C names; tensors are torch tensors on the current CUDA
device (torch supplies device memory and streams).  There is no fallback:
if libmoe.so is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID = 1
WS_STATUS_BYTES = 256

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_CUDA", 4: "MOE_ERR_DEVICE_INDEX", 5: "MOE_ERR_DEVICE_TIMEOUT",
                6: "MOE_ERR_WORKSPACE", 7: "MOE_ERR_PLACEMENT"}


class MoeError(RuntimeError):
    def __init__(self, call: str, status: int, info: Optional[int] = None):
        self.status = status
        self.info = info
        msg = f"{call}: {STATUS_NAMES.get(status, status)}"
        if info is not None:
            msg += f" (info={info})"
        super().__init__(msg)


class RouteCfg(ctypes.Structure):
    _fields_ = [("score_fn", ctypes.c_int32), ("k", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("group_topn", ctypes.c_int32)]


class FfnSchedule(ctypes.Structure):
    """moe_ffn_schedule: which CTA runs which FFN tile (never a row's bits).
    ph1_shift -1 = default; interleave and small_tiles 1 = default; cta_pairs
    1 runs tiles on pairs of SMs (0 = default)."""
    _fields_ = [("ph1_shift", ctypes.c_int32), ("interleave", ctypes.c_int32),
                ("small_tiles", ctypes.c_int32), ("cta_pairs", ctypes.c_int32)]

    def __init__(self, ph1_shift=-1, interleave=1, small_tiles=1, cta_pairs=0):
        super().__init__(ph1_shift, interleave, small_tiles, cta_pairs)


class PlacementC(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("n_ranks", ctypes.c_int32), ("ranks_per_node", ctypes.c_int32),
                ("slot_expert", ctypes.c_void_p), ("slot_rank", ctypes.c_void_p),
                ("rep_offsets", ctypes.c_void_p), ("rep_slots", ctypes.c_void_p),
                ("token_src_rank", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "moe_workspace_size": (_SZ, [_I64, _I32, _I32]),
    "moe_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "moe_check_device_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(_I32)]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [_P, _SZ, _I32, _P, _P]),
    "moe_prefetch_ffn_weights": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC), _P,
                                                _I32, _I32, _I64, _P]),
    "moe_route": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(RouteCfg), _P, _P, _P, _SZ, _P]),
    "moe_dispatch_layout": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC),
                                           _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_layout_noalloc": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC),
                                                   _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_replicas_workspace_size": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_route_replicas": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC), _I32, _I32,
                                          _P, _P, _P, _SZ, _P]),
    "moe_route_refine": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC), _P, _P, _P,
                                        _SZ, _P]),
    "moe_dispatch_layout_routed": (ctypes.c_int, [_P, _P, _I64, _I32, ctypes.POINTER(PlacementC),
                                                  _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P, _I32, _I32,
                                       _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_packed": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P, _I32, _I32,
                                              _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_gather": (ctypes.c_int, [_P, _I64, _I32, _P, _I64, _P, _P, _I32, _I32, _P,
                                              _P, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_pack_expert_weights": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_combine_merged": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(PlacementC), _I64, _I32,
                                          _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_balance_stats_layers": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "moe_balance_stats": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_layout_masked": (ctypes.c_int, [_P, _I64, _I32, ctypes.POINTER(PlacementC),
                                                  _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                                  _P]),
    "moe_permute_masked": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _I64, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_masked": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _I32, _P, _P, _I32, _I32,
                                              _P, _P, _P, _SZ, _P]),
    "moe_combine_masked": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I32, _I32, _P, _P, _P, _SZ,
                                          _P]),
    "moe_permute_fp8": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _I64, _P, _P, _P, _SZ, _P]),
    "moe_dequant_fp8": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_permute_shared": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_packed_shared": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P, _I32,
                                                     _I32, _I64, _I64, _I32, _P, _P, _P, _SZ,
                                                     _P]),
    "moe_grouped_ffn_packed_scheduled": (ctypes.c_int, [_P, _I64, _P, _P, _I32, _I32, _P, _P,
                                                        _I32, _I32, _I64, _I64, _I32,
                                                        ctypes.POINTER(FfnSchedule), _P, _P, _P,
                                                        _SZ, _P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_version": (ctypes.c_char_p, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so from this package directory (built by build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with grouped_ffn_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA tensor of {dtype}")


def _check(call: str, status: int):
    if status != MOE_OK:
        raise MoeError(call, status)


def _bf16(t: torch.Tensor, name: str):
    _need(t, torch.bfloat16, name)


# ------------------------------------------------------------------ workspace
def moe_workspace_size(T: int, k: int, n_slots: int) -> int:
    return int(lib().moe_workspace_size(T, k, n_slots))


def new_workspace(T: int, k: int, n_slots: int, device=None, stream=None,
                  n_experts: int = 0, n_ranks: int = 0) -> torch.Tensor:
    """Allocate (torch) and zero a workspace for calls on up to T tokens
    (large enough for replica routing too when n_experts and n_ranks are
    given)."""
    n = max(moe_workspace_size(T, k, n_slots), WS_STATUS_BYTES)
    if n_experts and n_ranks:
        n = max(n, moe_route_replicas_workspace_size(T, k, n_experts, n_slots, n_ranks))
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    moe_workspace_init(ws, stream)
    return ws


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check("moe_workspace_init", lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def moe_check_device_status(ws: torch.Tensor, stream=None):
    """Synchronise the stream; raise MoeError on a recorded device error."""
    info = _I32(0)
    st = lib().moe_check_device_status(_ptr(ws), _stream(stream), ctypes.byref(info))
    if st != MOE_OK:
        raise MoeError("device", st, info.value)


def moe_selftest_wait_timeout(ws: torch.Tensor, limit_us: int, waited_us=None, stream=None):
    """Run the device wait watchdog self-test (moe.h); the timeout it records
    is read with moe_check_device_status."""
    if waited_us is not None:
        _need(waited_us, torch.int32, "waited_us")
    _check("moe_selftest_wait_timeout",
           lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(limit_us),
                                           _ptr(waited_us), _stream(stream)))


# ------------------------------------------------------------------ placement
class DevicePlacement:
    """Placement tables on the device plus the C struct that points at them."""

    def __init__(self, slot_expert, slot_rank, rep_offsets, rep_slots, n_ranks: int,
                 ranks_per_node: int, token_src_rank=None, device="cuda"):
        def dev(a):
            return torch.as_tensor(a, dtype=torch.int32).to(device).contiguous()

        self.slot_expert = dev(slot_expert)
        self.slot_rank = dev(slot_rank)
        self.rep_offsets = dev(rep_offsets)
        self.rep_slots = dev(rep_slots)
        self.token_src_rank = None if token_src_rank is None else dev(token_src_rank)
        self.n_experts = int(self.rep_offsets.numel() - 1)
        self.n_slots = int(self.slot_expert.numel())
        self.n_ranks = int(n_ranks)
        self.ranks_per_node = int(ranks_per_node)
        self.c = PlacementC(self.n_experts, self.n_slots, self.n_ranks, self.ranks_per_node,
                            self.slot_expert.data_ptr(), self.slot_rank.data_ptr(),
                            self.rep_offsets.data_ptr(), self.rep_slots.data_ptr(),
                            None if self.token_src_rank is None else self.token_src_rank.data_ptr())

    @classmethod
    def from_tables(cls, pl, device="cuda"):
        """From any object with slot_expert, slot_rank, rep_offsets, rep_slots,
        n_ranks, ranks_per_node and token_src_rank attributes."""
        return cls(pl.slot_expert, pl.slot_rank, pl.rep_offsets, pl.rep_slots, pl.n_ranks,
                   pl.ranks_per_node, pl.token_src_rank, device)


# ------------------------------------------------------------------ calls
def moe_route(logits, cfg: RouteCfg, topk_ids, topk_w, ws=None, stream=None):
    _need(logits, torch.float32, "logits")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_w, torch.float32, "topk_w")
    T, E = logits.shape
    _check("moe_route", lib().moe_route(_ptr(logits), T, E, ctypes.byref(cfg), _ptr(topk_ids),
                                        _ptr(topk_w), _ptr(ws), 0 if ws is None else ws.numel(),
                                        _stream(stream)))


def moe_dispatch_layout(topk_ids, placement: DevicePlacement, slot, seg_counts, seg_offsets,
                        dest_row, src_assign, rank_counts, ws, stream=None):
    for n, t in (("topk_ids", topk_ids), ("slot", slot), ("seg_counts", seg_counts),
                 ("seg_offsets", seg_offsets), ("dest_row", dest_row),
                 ("src_assign", src_assign), ("rank_counts", rank_counts)):
        _need(t, torch.int32, n)
    T, k = topk_ids.shape
    _check("moe_dispatch_layout", lib().moe_dispatch_layout(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), _ptr(slot), _ptr(seg_counts),
        _ptr(seg_offsets), _ptr(dest_row), _ptr(src_assign), _ptr(rank_counts), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_prefetch_ffn_weights(topk_ids, placement: DevicePlacement, w_gate_up_packed, H: int,
                             I: int, max_bytes: int, stream=None):
    """Ask L2 for the weight tiles the grouped FFN's first wave streams first
    (moe.h); a hint that writes nothing."""
    _need(topk_ids, torch.int32, "topk_ids")
    _bf16(w_gate_up_packed, "w_gate_up_packed")
    T, k = topk_ids.shape
    _check("moe_prefetch_ffn_weights", lib().moe_prefetch_ffn_weights(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), _ptr(w_gate_up_packed), int(H), int(I),
        int(max_bytes), _stream(stream)))


def moe_dispatch_layout_noalloc(topk_ids, placement: DevicePlacement, slot, seg_counts,
                                seg_offsets, dest_row, src_assign, rank_counts, *, status,
                                stream=None):
    """The layout with the library's fixed device scratch instead of a
    workspace, for callers that cannot allocate.  `status` (required here) is
    a caller-owned device int32[3] that receives device-side errors; read it
    after the stream has run the call."""
    for n, t in (("topk_ids", topk_ids), ("slot", slot), ("seg_counts", seg_counts),
                 ("seg_offsets", seg_offsets), ("dest_row", dest_row),
                 ("src_assign", src_assign), ("rank_counts", rank_counts),
                 ("status", status)):
        _need(t, torch.int32, n)
    if status.numel() < 3:
        raise ValueError("moe_dispatch_layout_noalloc: status needs 3 int32 words")
    T, k = topk_ids.shape
    _check("moe_dispatch_layout_noalloc", lib().moe_dispatch_layout_noalloc(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), _ptr(slot), _ptr(seg_counts),
        _ptr(seg_offsets), _ptr(dest_row), _ptr(src_assign), _ptr(rank_counts), _ptr(status),
        _stream(stream)))


def moe_route_replicas_workspace_size(T: int, k: int, n_experts: int, n_slots: int,
                                      n_ranks: int) -> int:
    return int(lib().moe_route_replicas_workspace_size(T, k, n_experts, n_slots, n_ranks))


def moe_route_replicas(topk_ids, placement: DevicePlacement, c_num: int, c_den: int, slot,
                       inter_node, ws, stream=None):
    """Locality-preferred replica choice per assignment (water-filling under
    load bounds C = c_num / c_den); inter_node is a device int32[1]."""
    _need(topk_ids, torch.int32, "topk_ids")
    _need(slot, torch.int32, "slot")
    _need(inter_node, torch.int32, "inter_node")
    T, k = topk_ids.shape
    _check("moe_route_replicas", lib().moe_route_replicas(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), c_num, c_den, _ptr(slot),
        _ptr(inter_node), _ptr(ws), ws.numel(), _stream(stream)))


def moe_route_refine(topk_ids, placement: DevicePlacement, slot, messages, ws, stream=None):
    """Consolidate each token's remote requests onto fewer nodes, in place on
    slot (same per-copy counts); messages is a device int32[2] that receives
    the (token, remote node) pairs before and after."""
    _need(topk_ids, torch.int32, "topk_ids")
    _need(slot, torch.int32, "slot")
    _need(messages, torch.int32, "messages")
    T, k = topk_ids.shape
    _check("moe_route_refine", lib().moe_route_refine(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), _ptr(slot), _ptr(messages), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_dispatch_layout_routed(topk_ids, slot_in, placement: DevicePlacement, seg_counts,
                               seg_offsets, dest_row, src_assign, rank_counts, ws, stream=None):
    for n, t in (("topk_ids", topk_ids), ("slot_in", slot_in), ("seg_counts", seg_counts),
                 ("seg_offsets", seg_offsets), ("dest_row", dest_row),
                 ("src_assign", src_assign), ("rank_counts", rank_counts)):
        _need(t, torch.int32, n)
    T, k = topk_ids.shape
    _check("moe_dispatch_layout_routed", lib().moe_dispatch_layout_routed(
        _ptr(topk_ids), _ptr(slot_in), T, k, ctypes.byref(placement.c), _ptr(seg_counts),
        _ptr(seg_offsets), _ptr(dest_row), _ptr(src_assign), _ptr(rank_counts), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_permute(x, k: int, dest_row, x_perm, ws, stream=None):
    _bf16(x, "x")
    _bf16(x_perm, "x_perm")
    _need(dest_row, torch.int32, "dest_row")
    T, H = x.shape
    _check("moe_permute", lib().moe_permute(_ptr(x), T, H, k, _ptr(dest_row), _ptr(x_perm),
                                            _ptr(ws), ws.numel(), _stream(stream)))


def moe_grouped_ffn(x_perm, seg_offsets, seg_expert, w_gate_up, w_down, h, y_perm, ws,
                    stream=None):
    for n, t in (("x_perm", x_perm), ("w_gate_up", w_gate_up), ("w_down", w_down),
                 ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(seg_offsets, torch.int32, "seg_offsets")
    _need(seg_expert, torch.int32, "seg_expert")
    n_rows, H = x_perm.shape
    E, two_i, H2 = w_gate_up.shape
    I = two_i // 2
    if H2 != H or tuple(w_down.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) \
            or tuple(y_perm.shape) != (n_rows, H):
        raise ValueError("moe_grouped_ffn: inconsistent shapes")
    S = seg_expert.numel()
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(
        _ptr(x_perm), n_rows, _ptr(seg_offsets), _ptr(seg_expert), S, E, _ptr(w_gate_up),
        _ptr(w_down), H, I, _ptr(h), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_grouped_ffn_packed(x_perm, seg_offsets, seg_expert, w_gate_up_packed, w_down_packed,
                           h, y_perm, ws, stream=None):
    """moe_grouped_ffn on weights packed by moe_pack_expert_weights (same
    shapes as the plain [E,2I,H] and [E,H,I] tensors)."""
    for n, t in (("x_perm", x_perm), ("w_gate_up_packed", w_gate_up_packed),
                 ("w_down_packed", w_down_packed), ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(seg_offsets, torch.int32, "seg_offsets")
    _need(seg_expert, torch.int32, "seg_expert")
    n_rows, H = x_perm.shape
    E, two_i, H2 = w_gate_up_packed.shape
    I = two_i // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) \
            or tuple(y_perm.shape) != (n_rows, H):
        raise ValueError("moe_grouped_ffn_packed: inconsistent shapes")
    S = seg_expert.numel()
    _check("moe_grouped_ffn_packed", lib().moe_grouped_ffn_packed(
        _ptr(x_perm), n_rows, _ptr(seg_offsets), _ptr(seg_expert), S, E, _ptr(w_gate_up_packed),
        _ptr(w_down_packed), H, I, _ptr(h), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_grouped_ffn_gather(x, k: int, src_assign, seg_offsets, seg_expert, w_gate_up_packed,
                           w_down_packed, h, y_perm, ws, stream=None):
    """The grouped FFN reading its gate/up rows straight from x through
    src_assign (TMA gather), with packed weights; no permuted copy."""
    for n, t in (("x", x), ("w_gate_up_packed", w_gate_up_packed),
                 ("w_down_packed", w_down_packed), ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(src_assign, torch.int32, "src_assign")
    _need(seg_offsets, torch.int32, "seg_offsets")
    _need(seg_expert, torch.int32, "seg_expert")
    T, H = x.shape
    n_rows = y_perm.shape[0]
    E, two_i, H2 = w_gate_up_packed.shape
    I = two_i // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) \
            or src_assign.numel() < n_rows:
        raise ValueError("moe_grouped_ffn_gather: inconsistent shapes")
    _check("moe_grouped_ffn_gather", lib().moe_grouped_ffn_gather(
        _ptr(x), T, k, _ptr(src_assign), n_rows, _ptr(seg_offsets), _ptr(seg_expert),
        seg_expert.numel(), E, _ptr(w_gate_up_packed), _ptr(w_down_packed), H, I, _ptr(h),
        _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_pack_expert_weights(w_gate_up, w_down, w_gate_up_packed, w_down_packed, stream=None):
    """Rearrange [E,2I,H] / [E,H,I] expert weights into the library's
    tile-contiguous layout (outputs have the same shapes)."""
    for n, t in (("w_gate_up", w_gate_up), ("w_down", w_down),
                 ("w_gate_up_packed", w_gate_up_packed), ("w_down_packed", w_down_packed)):
        _bf16(t, n)
    E, two_i, H = w_gate_up.shape
    I = two_i // 2
    if tuple(w_down.shape) != (E, H, I) or w_gate_up_packed.shape != w_gate_up.shape \
            or w_down_packed.shape != w_down.shape:
        raise ValueError("moe_pack_expert_weights: inconsistent shapes")
    _check("moe_pack_expert_weights", lib().moe_pack_expert_weights(
        _ptr(w_gate_up), _ptr(w_down), E, H, I, _ptr(w_gate_up_packed), _ptr(w_down_packed),
        _stream(stream)))


def moe_combine(y_perm, dest_row, topk_w, y, ws, shared=None, stream=None):
    _bf16(y_perm, "y_perm")
    _bf16(y, "y")
    if shared is not None:
        _bf16(shared, "shared")
    _need(dest_row, torch.int32, "dest_row")
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    H = y.shape[1]
    _check("moe_combine", lib().moe_combine(_ptr(y_perm), _ptr(dest_row), _ptr(topk_w), T, k, H,
                                            _ptr(shared), _ptr(y), _ptr(ws), ws.numel(),
                                            _stream(stream)))


def moe_combine_merged(y_perm, dest_row, topk_w, slot, placement: DevicePlacement, y, messages,
                       ws, shared=None, stream=None):
    """Combine with node-local pre-reduction; messages (device int32[2])
    receives the inter-node dispatch messages before and after merge."""
    _bf16(y_perm, "y_perm")
    _bf16(y, "y")
    if shared is not None:
        _bf16(shared, "shared")
    for n, t in (("dest_row", dest_row), ("slot", slot), ("messages", messages)):
        _need(t, torch.int32, n)
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    _check("moe_combine_merged", lib().moe_combine_merged(
        _ptr(y_perm), _ptr(dest_row), _ptr(topk_w), _ptr(slot), ctypes.byref(placement.c), T, k,
        y.shape[1], _ptr(shared), _ptr(y), _ptr(messages), _ptr(ws), ws.numel(), _stream(stream)))


def moe_balance_stats_layers(rank_counts, balancedness, max_sum, total, stream=None):
    """Balancedness over layers: rank_counts int32 [L, R]; outputs device
    float64[1], int64[1], int64[1]."""
    _need(rank_counts, torch.int32, "rank_counts")
    _need(balancedness, torch.float64, "balancedness")
    _need(max_sum, torch.int64, "max_sum")
    _need(total, torch.int64, "total")
    L, R = rank_counts.shape
    _check("moe_balance_stats_layers", lib().moe_balance_stats_layers(
        _ptr(rank_counts), L, R, _ptr(balancedness), _ptr(max_sum), _ptr(total),
        _stream(stream)))


def moe_balance_stats(rank_counts, balancedness, max_count, total, ws=None, stream=None):
    _need(rank_counts, torch.int32, "rank_counts")
    _need(balancedness, torch.float64, "balancedness")
    _need(max_count, torch.int32, "max_count")
    _need(total, torch.int64, "total")
    _check("moe_balance_stats", lib().moe_balance_stats(
        _ptr(rank_counts), rank_counts.numel(), _ptr(balancedness), _ptr(max_count), _ptr(total),
        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


# ------------------------------------------------------------------ shared expert in the routed launch
def moe_permute_shared(x, k: int, dest_row, x_perm, ws, stream=None):
    """moe_permute plus a copy of every token row t at row T*k + t
    (x_perm has T*k + T rows)."""
    _bf16(x, "x")
    _bf16(x_perm, "x_perm")
    _need(dest_row, torch.int32, "dest_row")
    T, H = x.shape
    if x_perm.shape[0] < T * k + T:
        raise ValueError("moe_permute_shared: x_perm needs T*k + T rows")
    _check("moe_permute_shared", lib().moe_permute_shared(
        _ptr(x), T, H, k, _ptr(dest_row), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_grouped_ffn_packed_shared(x_perm, seg_offsets, seg_expert, w_gate_up_packed,
                                  w_down_packed, shared_row0: int, shared_rows: int,
                                  shared_expert: int, h, y_perm, ws, stream=None):
    """moe_grouped_ffn_packed plus one segment [shared_row0, shared_row0 +
    shared_rows) run with expert shared_expert in the same launch."""
    for n, t in (("x_perm", x_perm), ("w_gate_up_packed", w_gate_up_packed),
                 ("w_down_packed", w_down_packed), ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(seg_offsets, torch.int32, "seg_offsets")
    _need(seg_expert, torch.int32, "seg_expert")
    n_rows, H = x_perm.shape
    E, two_i, H2 = w_gate_up_packed.shape
    I = two_i // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) \
            or tuple(y_perm.shape) != (n_rows, H):
        raise ValueError("moe_grouped_ffn_packed_shared: inconsistent shapes")
    _check("moe_grouped_ffn_packed_shared", lib().moe_grouped_ffn_packed_shared(
        _ptr(x_perm), n_rows, _ptr(seg_offsets), _ptr(seg_expert), seg_expert.numel(), E,
        _ptr(w_gate_up_packed), _ptr(w_down_packed), H, I, shared_row0, shared_rows,
        shared_expert, _ptr(h), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_grouped_ffn_packed_scheduled(x_perm, seg_offsets, seg_expert, w_gate_up_packed,
                                     w_down_packed, shared_row0: int, shared_rows: int,
                                     shared_expert: int, schedule: FfnSchedule, h, y_perm, ws,
                                     stream=None):
    """moe_grouped_ffn_packed_shared with an explicit tile schedule."""
    for n, t in (("x_perm", x_perm), ("w_gate_up_packed", w_gate_up_packed),
                 ("w_down_packed", w_down_packed), ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(seg_offsets, torch.int32, "seg_offsets")
    _need(seg_expert, torch.int32, "seg_expert")
    n_rows, H = x_perm.shape
    E, two_i, H2 = w_gate_up_packed.shape
    I = two_i // 2
    if H2 != H or tuple(w_down_packed.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) \
            or tuple(y_perm.shape) != (n_rows, H):
        raise ValueError("moe_grouped_ffn_packed_scheduled: inconsistent shapes")
    _check("moe_grouped_ffn_packed_scheduled", lib().moe_grouped_ffn_packed_scheduled(
        _ptr(x_perm), n_rows, _ptr(seg_offsets), _ptr(seg_expert), seg_expert.numel(), E,
        _ptr(w_gate_up_packed), _ptr(w_down_packed), H, I, shared_row0, shared_rows,
        shared_expert, None if schedule is None else ctypes.byref(schedule), _ptr(h),
        _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


# ------------------------------------------------------------------ fixed-capacity layout
def moe_dispatch_layout_masked(topk_ids, placement: DevicePlacement, cap: int, slot, seg_counts,
                               masked_m, dest_row, src_assign, rank_counts, n_dropped, ws,
                               stream=None):
    """Fixed-capacity layout: slot s owns rows [s*cap, (s+1)*cap); its
    assignments past the first `cap` are dropped (dest_row -1).  src_assign
    has S*cap entries; n_dropped is a device int32[1]."""
    for n, t in (("topk_ids", topk_ids), ("slot", slot), ("seg_counts", seg_counts),
                 ("masked_m", masked_m), ("dest_row", dest_row), ("src_assign", src_assign),
                 ("rank_counts", rank_counts), ("n_dropped", n_dropped)):
        _need(t, torch.int32, n)
    T, k = topk_ids.shape
    if src_assign.numel() < placement.c.n_slots * cap:
        raise ValueError("moe_dispatch_layout_masked: src_assign needs S*cap entries")
    _check("moe_dispatch_layout_masked", lib().moe_dispatch_layout_masked(
        _ptr(topk_ids), T, k, ctypes.byref(placement.c), cap, _ptr(slot), _ptr(seg_counts),
        _ptr(masked_m), _ptr(dest_row), _ptr(src_assign), _ptr(rank_counts), _ptr(n_dropped),
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_permute_masked(x, k: int, dest_row, x_perm, ws, stream=None):
    """moe_permute into x_perm [n_rows, H] where dest_row -1 is a drop."""
    _bf16(x, "x")
    _bf16(x_perm, "x_perm")
    _need(dest_row, torch.int32, "dest_row")
    T, H = x.shape
    _check("moe_permute_masked", lib().moe_permute_masked(
        _ptr(x), T, H, k, _ptr(dest_row), x_perm.shape[0], _ptr(x_perm), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_grouped_ffn_masked(x_perm, cap: int, masked_m, seg_expert, w_gate_up_packed,
                           w_down_packed, h, y_perm, ws, stream=None):
    """The grouped FFN on a fixed-capacity layout (packed weights): slot s
    is rows [s*cap, s*cap + masked_m[s]) of x_perm [S*cap, H]."""
    for n, t in (("x_perm", x_perm), ("w_gate_up_packed", w_gate_up_packed),
                 ("w_down_packed", w_down_packed), ("h", h), ("y_perm", y_perm)):
        _bf16(t, n)
    _need(masked_m, torch.int32, "masked_m")
    _need(seg_expert, torch.int32, "seg_expert")
    S = seg_expert.numel()
    n_rows, H = x_perm.shape
    E, two_i, H2 = w_gate_up_packed.shape
    I = two_i // 2
    if n_rows != S * cap or masked_m.numel() != S or H2 != H or \
            tuple(w_down_packed.shape) != (E, H, I) or tuple(h.shape) != (n_rows, I) or \
            tuple(y_perm.shape) != (n_rows, H):
        raise ValueError("moe_grouped_ffn_masked: inconsistent shapes")
    _check("moe_grouped_ffn_masked", lib().moe_grouped_ffn_masked(
        _ptr(x_perm), cap, _ptr(masked_m), _ptr(seg_expert), S, E, _ptr(w_gate_up_packed),
        _ptr(w_down_packed), H, I, _ptr(h), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def moe_combine_masked(y_perm, dest_row, topk_w, y, ws, shared=None, stream=None):
    """moe_combine over y_perm [n_rows, H] where dest_row -1 (a dropped
    assignment) adds nothing."""
    _bf16(y_perm, "y_perm")
    _bf16(y, "y")
    if shared is not None:
        _bf16(shared, "shared")
    _need(dest_row, torch.int32, "dest_row")
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    _check("moe_combine_masked", lib().moe_combine_masked(
        _ptr(y_perm), y_perm.shape[0], _ptr(dest_row), _ptr(topk_w), T, k, y.shape[1],
        _ptr(shared), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


# ------------------------------------------------------------------ FP8 dispatch
def moe_permute_fp8(x, k: int, dest_row, xq, x_scale, ws, stream=None):
    """Quantize each token row to E4M3 (power-of-two scale per 128
    channels) and write it to its k dispatched rows: xq uint8 [n_rows, H],
    x_scale fp32 [n_rows, H/128]; dest_row -1 is a drop."""
    _bf16(x, "x")
    _need(dest_row, torch.int32, "dest_row")
    _need(xq, torch.uint8, "xq")
    _need(x_scale, torch.float32, "x_scale")
    T, H = x.shape
    n_rows = xq.shape[0]
    if xq.shape[1] != H or tuple(x_scale.shape) != (n_rows, H // 128):
        raise ValueError("moe_permute_fp8: inconsistent shapes")
    _check("moe_permute_fp8", lib().moe_permute_fp8(
        _ptr(x), T, H, k, _ptr(dest_row), n_rows, _ptr(xq), _ptr(x_scale), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_dequant_fp8(xq, x_scale, x_perm, masked_m=None, cap: int = 0, ws=None, stream=None):
    """x_perm = bf16(E4M3(xq) * x_scale); with masked_m only the used rows of
    each fixed-capacity slot."""
    _need(xq, torch.uint8, "xq")
    _need(x_scale, torch.float32, "x_scale")
    _bf16(x_perm, "x_perm")
    if masked_m is not None:
        _need(masked_m, torch.int32, "masked_m")
    n_rows, H = xq.shape
    if tuple(x_perm.shape) != (n_rows, H) or tuple(x_scale.shape) != (n_rows, H // 128):
        raise ValueError("moe_dequant_fp8: inconsistent shapes")
    _check("moe_dequant_fp8", lib().moe_dequant_fp8(
        _ptr(xq), _ptr(x_scale), n_rows, H, cap, _ptr(masked_m), _ptr(x_perm), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_version() -> str:
    return lib().moe_version().decode()
