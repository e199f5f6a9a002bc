"""MoELayer: the whole hot path as one call over persistent device buffers.

route -> dispatch_layout -> permute -> grouped_ffn (+ shared expert) ->
combine -> balance_stats, each a libmoe.so kernel launch on one stream, with
no host synchronisation inside a step (the host never reads segment sizes:
they stay on the device, as "Zepp" Section 6.4 notes for planning without
per-layer host sync).  Buffers are allocated once, for the largest token
count, through torch; the library itself allocates nothing.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import moe


class MoELayer:
    PREFETCH_BYTES = 96 << 20          # three quarters of L2
    PREFETCH_MAX_DISPATCH = 32 << 20   # dispatched bf16 bytes up to which it applies

    def __init__(self, *, H: int, I: int, E: int, k: int, placement: moe.DevicePlacement,
                 w_gate_up: torch.Tensor, w_down: torch.Tensor, max_tokens: int,
                 score_fn: int = moe.MOE_SCORE_SOFTMAX, n_groups: int = 1,
                 topk_groups: int = 1, group_topn: int = 1,
                 shared_w_gate_up: Optional[torch.Tensor] = None,
                 shared_w_down: Optional[torch.Tensor] = None, device="cuda",
                 packed: bool = True, replica_relax: Optional[tuple] = None,
                 replica_refine: bool = False, gather: bool = False,
                 masked_cap: Optional[int] = None,
                 fp8_dispatch: bool = False, fuse_shared: bool = True,
                 ffn_schedule: Optional[moe.FfnSchedule] = None):
        """replica_relax=(c_num, c_den) chooses each assignment's replica by
        locality-preferred water-filling with load bounds C = c_num/c_den
        (moe_route_replicas); None keeps the fixed replica rule.
        replica_refine=True then consolidates each token's remote requests
        onto fewer nodes with the same per-copy counts (moe_route_refine);
        `messages` holds the (token, remote node) pairs before and after.
        gather=True reads the FFN's rows straight from x through the
        inverse permutation (moe_grouped_ffn_gather): no permute step.
        masked_cap=c uses the fixed-capacity layout (moe_dispatch_layout_masked):
        every slot owns c rows, assignments beyond them are dropped.
        fp8_dispatch=True moves E4M3 codes and block scales through the
        dispatched buffer (moe_permute_fp8) and restores bf16 rows before
        the FFN (moe_dequant_fp8).
        fuse_shared=True runs a shared expert of the routed experts' width
        inside the routed experts' FFN launch (moe_permute_shared +
        moe_grouped_ffn_packed_shared) in the plain contiguous bf16 step;
        otherwise it is a second launch.  The results are the same bits.
        ffn_schedule (packed weights, contiguous layout) sets the grouped
        FFN's tile schedule; None is the library's default.  Every schedule
        gives the same bits."""
        if (gather or masked_cap is not None) and not packed:
            raise ValueError("gather and fixed-capacity modes stream packed weights")
        if gather and (masked_cap is not None or fp8_dispatch):
            raise ValueError("gather mode reads x directly: no fixed capacity, no FP8 dispatch")
        if masked_cap is not None and (replica_relax is not None or masked_cap < 1):
            raise ValueError("fixed-capacity layout: cap >= 1, fixed replica rule")
        if ffn_schedule is not None and (not packed or gather or masked_cap is not None):
            raise ValueError("ffn_schedule applies to the packed contiguous FFN")
        self.ffn_schedule = ffn_schedule
        self.gather = gather
        self.masked_cap = masked_cap
        self.fp8_dispatch = fp8_dispatch
        self.H, self.I, self.E, self.k = H, I, E, k
        self.placement = placement
        self.packed = packed
        self.fuse_shared = bool(
            fuse_shared and shared_w_gate_up is not None and packed and not gather
            and masked_cap is None and not fp8_dispatch
            and tuple(shared_w_gate_up.shape[1:]) == (2 * I, H))
        if self.fuse_shared:
            # one packed tensor holds the routed experts and, as expert E,
            # the shared one, so that one launch serves both
            gu = torch.empty((E + 1, 2 * I, H), dtype=w_gate_up.dtype, device=w_gate_up.device)
            dn = torch.empty((E + 1, H, I), dtype=w_down.dtype, device=w_down.device)
            moe.moe_pack_expert_weights(w_gate_up, w_down, gu[:E], dn[:E])
            moe.moe_pack_expert_weights(shared_w_gate_up, shared_w_down, gu[E:], dn[E:])
            w_gate_up, w_down = gu, dn
            shared_w_gate_up = shared_w_down = None
            self.shared_I = I
        elif packed:
            # one-time rearrangement into the tile-contiguous layout the FFN
            # kernel streams best (each TMA box is one contiguous block)
            w_gate_up, w_down = self._pack(w_gate_up, w_down)
            if shared_w_gate_up is not None:
                shared_w_gate_up, shared_w_down = self._pack(shared_w_gate_up, shared_w_down)
        self.w_gate_up, self.w_down = w_gate_up, w_down
        self.shared_w_gate_up, self.shared_w_down = shared_w_gate_up, shared_w_down
        self.cfg = moe.RouteCfg(score_fn, k, n_groups, topk_groups, group_topn)
        self.max_tokens = max_tokens
        dev = torch.device(device)
        A = max_tokens * k
        S, R = placement.n_slots, placement.n_ranks
        i32 = dict(dtype=torch.int32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.topk_ids = torch.empty(max_tokens, k, **i32)
        self.topk_w = torch.empty(max_tokens, k, dtype=torch.float32, device=dev)
        # dispatched rows: T*k in the contiguous layout (+ T for a fused
        # shared expert), S*cap in the fixed one
        rows = A if masked_cap is None else S * masked_cap
        if self.fuse_shared:
            rows = A + max_tokens
        self.slot = torch.empty(A, **i32)
        self.seg_counts = torch.empty(S, **i32)
        self.seg_offsets = torch.empty(S + 1, **i32)
        self.dest_row = torch.empty(A, **i32)
        self.src_assign = torch.empty(rows, **i32)
        self.rank_counts = torch.empty(R, **i32)
        self.masked_m = torch.zeros(S, **i32)
        self.n_dropped = torch.zeros(1, **i32)
        self.x_perm = torch.empty(0 if gather else rows, H, **bf)
        if fp8_dispatch:
            self.xq = torch.empty(rows, H, dtype=torch.uint8, device=dev)
            self.x_scale = torch.empty(rows, H // 128, dtype=torch.float32, device=dev)
        self.h = torch.empty(rows, I, **bf)
        self.y_perm = torch.empty(rows, H, **bf)
        self.balancedness = torch.empty(1, dtype=torch.float64, device=dev)
        self.max_count = torch.empty(1, **i32)
        self.total = torch.empty(1, dtype=torch.int64, device=dev)
        self.ws = moe.new_workspace(max_tokens, k, S, device=dev, n_experts=E, n_ranks=R)
        # the balancedness statistic needs only the layout's per-rank counts:
        # it runs on a side stream forked after the layout and joined at the
        # end of the step, off the permute -> FFN -> combine path
        self._side = torch.cuda.Stream(device=dev)
        self._ev_layout = torch.cuda.Event()
        self._ev_stats = torch.cuda.Event()
        self.replica_relax = replica_relax
        if replica_refine and replica_relax is None:
            raise ValueError("replica_refine refines the water-filling routing (replica_relax)")
        self.replica_refine = replica_refine
        self.inter_node = torch.zeros(1, **i32)
        self.messages = torch.zeros(2, **i32)
        if self.fuse_shared:
            pass
        elif shared_w_gate_up is not None:
            self.shared_I = shared_w_gate_up.shape[1] // 2
            self.shared_h = torch.empty(max_tokens, self.shared_I, **bf)
            self.shared_y = torch.empty(max_tokens, H, **bf)
            self.shared_expert = torch.zeros(1, **i32)
            self._shared_offsets = {}
        else:
            self.shared_I = 0
        # per step: route, layout scan + finalize, permute, FFN, combine,
        # balance (+1 shared FFN, +4 replica routing: prep, key scan,
        # water-fill, assign, +1 refinement, +1 FP8 dequantization, +1
        # weight prefetch);
        # packing happens once, here
        # L2 prefetch of the FFN's first weight tiles, on the side stream
        # right after routing: worth it when the step is weight-bound and its
        # dispatch is small (decode), so that the fetched tiles are neither
        # competing with nor evicted by a large permute; exact placement
        # without replicas, packed weights, the contiguous layout
        small = max_tokens * k * H * 2 <= self.PREFETCH_MAX_DISPATCH
        self.prefetch_bytes = self.PREFETCH_BYTES if (
            small and packed and not gather and masked_cap is None and replica_relax is None
            and placement.n_slots == placement.n_experts) else 0
        self._ev_route = torch.cuda.Event()
        # the layout scan takes up to 1024 assignments in one CTA, which then
        # also finalizes (no second launch) on the contiguous layout
        one_tile = max_tokens * k <= 1024 and masked_cap is None
        self.launches_per_step = 7 + (1 if shared_w_gate_up is not None else 0) + \
            (4 if replica_relax is not None else 0) + (1 if replica_refine else 0) - \
            (1 if gather else 0) + \
            (1 if fp8_dispatch else 0) + (1 if self.prefetch_bytes else 0) - (1 if one_tile else 0)

    @staticmethod
    def _pack(w_gate_up, w_down):
        gu, d = torch.empty_like(w_gate_up), torch.empty_like(w_down)
        moe.moe_pack_expert_weights(w_gate_up, w_down, gu, d)
        return gu, d

    def _ffn(self, x_perm, offs, experts, wgu, wd, h, y, ws, stream):
        if self.ffn_schedule is not None:
            moe.moe_grouped_ffn_packed_scheduled(x_perm, offs, experts, wgu, wd, 0, 0, 0,
                                                 self.ffn_schedule, h, y, ws, stream)
        elif self.packed:
            moe.moe_grouped_ffn_packed(x_perm, offs, experts, wgu, wd, h, y, ws, stream)
        else:
            moe.moe_grouped_ffn(x_perm, offs, experts, wgu, wd, h, y, ws, stream)

    def _shared_offs(self, T: int) -> torch.Tensor:
        t = self._shared_offsets.get(T)
        if t is None:
            t = torch.tensor([0, T], dtype=torch.int32).to(self.shared_expert.device)
            self._shared_offsets[T] = t
        return t

    def forward(self, logits: torch.Tensor, x: torch.Tensor, y: torch.Tensor, stream=None,
                mark=None):
        """One step on device-resident inputs; y [T,H] bf16 is written.
        mark(name), if given, is called after each stage is enqueued (the
        benchmark records a CUDA event there)."""
        mark = mark or (lambda name: None)
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError("more tokens than the layer was sized for")
        A = T * self.k
        ids, w = self.topk_ids[:T], self.topk_w[:T]
        moe.moe_route(logits, self.cfg, ids, w, self.ws, stream)
        self._fork_prefetch(ids, stream)
        mark("route")
        if self.masked_cap is not None:
            return self._forward_masked(x, y, ids, w, T, A, stream, mark)
        if self.replica_relax is None:
            moe.moe_dispatch_layout(ids, self.placement, self.slot[:A], self.seg_counts,
                                    self.seg_offsets, self.dest_row[:A], self.src_assign[:A],
                                    self.rank_counts, self.ws, stream)
        else:
            moe.moe_route_replicas(ids, self.placement, *self.replica_relax, self.slot[:A],
                                   self.inter_node, self.ws, stream)
            if self.replica_refine:
                moe.moe_route_refine(ids, self.placement, self.slot[:A], self.messages, self.ws,
                                     stream)
            moe.moe_dispatch_layout_routed(ids, self.slot[:A], self.placement, self.seg_counts,
                                           self.seg_offsets, self.dest_row[:A],
                                           self.src_assign[:A], self.rank_counts, self.ws, stream)
        mark("layout")
        self._fork_balance(stream)
        if self.gather:
            mark("permute")
            moe.moe_grouped_ffn_gather(x, self.k, self.src_assign[:A], self.seg_offsets,
                                       self.placement.slot_expert, self.w_gate_up, self.w_down,
                                       self.h[:A], self.y_perm[:A], self.ws, stream)
        elif self.fuse_shared:
            # rows [A, A + T) carry the tokens once more for the shared
            # expert (expert E of the packed weights), in the same launch
            moe.moe_permute_shared(x, self.k, self.dest_row[:A], self.x_perm[:A + T], self.ws,
                                   stream)
            mark("permute")
            if self.ffn_schedule is not None:
                moe.moe_grouped_ffn_packed_scheduled(
                    self.x_perm[:A + T], self.seg_offsets, self.placement.slot_expert,
                    self.w_gate_up, self.w_down, A, T, self.E, self.ffn_schedule,
                    self.h[:A + T], self.y_perm[:A + T], self.ws, stream)
            else:
                moe.moe_grouped_ffn_packed_shared(self.x_perm[:A + T], self.seg_offsets,
                                                  self.placement.slot_expert, self.w_gate_up,
                                                  self.w_down, A, T, self.E, self.h[:A + T],
                                                  self.y_perm[:A + T], self.ws, stream)
        else:
            self._dispatch(x, A, A, None, stream, mark)
            self._ffn(self.x_perm[:A], self.seg_offsets, self.placement.slot_expert,
                      self.w_gate_up, self.w_down, self.h[:A], self.y_perm[:A], self.ws, stream)
        mark("grouped_ffn")
        shared = self.shared_output(T) if self.fuse_shared else self._shared(x, T, stream, mark)
        moe.moe_combine(self.y_perm[:A], self.dest_row[:A], w, y, self.ws, shared, stream)
        mark("combine")
        self._join_balance(stream, mark)
        return y

    def _dispatch(self, x, A, rows, masked_m, stream, mark):
        """Rows of x into the dispatched buffer: a bf16 copy, or E4M3 codes
        plus block scales restored to bf16 by the receiving step."""
        dr = self.dest_row[:A]
        if self.fp8_dispatch:
            moe.moe_permute_fp8(x, self.k, dr, self.xq[:rows], self.x_scale[:rows], self.ws, stream)
            mark("permute")
            moe.moe_dequant_fp8(self.xq[:rows], self.x_scale[:rows], self.x_perm[:rows], masked_m,
                                self.masked_cap or 0, self.ws, stream)
            mark("dequant")
        elif masked_m is not None:
            moe.moe_permute_masked(x, self.k, dr, self.x_perm[:rows], self.ws, stream)
            mark("permute")
        else:
            moe.moe_permute(x, self.k, dr, self.x_perm[:A], self.ws, stream)
            mark("permute")

    def _shared(self, x, T, stream, mark):
        if not self.shared_I:
            return None
        self._ffn(x, self._shared_offs(T), self.shared_expert, self.shared_w_gate_up,
                  self.shared_w_down, self.shared_h[:T], self.shared_y[:T], self.ws, stream)
        mark("shared_ffn")
        return self.shared_y[:T]

    def shared_output(self, T: int):
        """The shared expert's output rows [T, H] of the last step, or None
        when the layer has no shared expert."""
        if self.fuse_shared:
            A = T * self.k
            return self.y_perm[A:A + T]
        return self.shared_y[:T] if self.shared_I else None

    def _fork_prefetch(self, ids, stream):
        """The routed ids fix which weight tiles the FFN streams first: ask
        L2 for them on the side stream while the layout and the permute run."""
        if not self.prefetch_bytes:
            return
        s = stream or torch.cuda.current_stream()
        self._ev_route.record(s)
        self._side.wait_event(self._ev_route)
        moe.moe_prefetch_ffn_weights(ids, self.placement, self.w_gate_up, self.H, self.I,
                                     self.prefetch_bytes, self._side)

    def _fork_balance(self, stream):
        s = stream or torch.cuda.current_stream()
        self._ev_layout.record(s)
        self._side.wait_event(self._ev_layout)
        moe.moe_balance_stats(self.rank_counts, self.balancedness, self.max_count, self.total,
                              None, self._side)
        self._ev_stats.record(self._side)

    def _join_balance(self, stream, mark):
        (stream or torch.cuda.current_stream()).wait_event(self._ev_stats)
        mark("balance")

    def _forward_masked(self, x, y, ids, w, T, A, stream, mark):
        """The step on the fixed-capacity layout: every buffer and launch has
        the same shape whatever the routing; dropped assignments add
        nothing to y."""
        cap = self.masked_cap
        rows = self.placement.n_slots * cap
        moe.moe_dispatch_layout_masked(ids, self.placement, cap, self.slot[:A], self.seg_counts,
                                       self.masked_m, self.dest_row[:A], self.src_assign,
                                       self.rank_counts, self.n_dropped, self.ws, stream)
        mark("layout")
        self._fork_balance(stream)
        self._dispatch(x, A, rows, self.masked_m, stream, mark)
        moe.moe_grouped_ffn_masked(self.x_perm, cap, self.masked_m, self.placement.slot_expert,
                                   self.w_gate_up, self.w_down, self.h, self.y_perm, self.ws,
                                   stream)
        mark("grouped_ffn")
        shared = self._shared(x, T, stream, mark)
        moe.moe_combine_masked(self.y_perm, self.dest_row[:A], w, y, self.ws, shared, stream)
        mark("combine")
        self._join_balance(stream, mark)
        return y

    def capture(self, logits: torch.Tensor, x: torch.Tensor, y: torch.Tensor):
        """Record one whole step (every kernel of forward) as a CUDA graph
        over these fixed buffers and return it; graph.replay() then reruns
        the step on whatever the buffers hold, with one launch from the
        host.  Segment sizes never reach the host, so the dynamic
        contiguous layout needs no padding to be replayable.  Call forward
        once first (per-device set-up happens on the first call)."""
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream(device=y.device)
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                self.forward(logits, x, y, torch.cuda.current_stream())
        torch.cuda.current_stream().wait_stream(stream)
        return graph

    def forward_host(self, logits_host: torch.Tensor, x_host: torch.Tensor,
                     y_host: torch.Tensor, logits_dev: torch.Tensor, x_dev: torch.Tensor,
                     y_dev: torch.Tensor, stream=None):
        """End to end from pinned host memory: copy the step's inputs in, run
        the layer, copy the output back (asynchronous on the stream)."""
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            logits_dev.copy_(logits_host, non_blocking=True)
            x_dev.copy_(x_host, non_blocking=True)
            self.forward(logits_dev, x_dev, y_dev, s)
            y_host.copy_(y_dev, non_blocking=True)
        return y_host

    def check(self, stream=None):
        """Raise MoeError if any kernel recorded a device-side error."""
        moe.moe_check_device_status(self.ws, stream)


class HostPipeline:
    """Steps fed from pinned host memory with the copies overlapped.

    Step i copies its inputs host->device on one stream, runs the layer on a
    second, and copies its output back on a third; `depth` sets of device
    input/output buffers let step i+1's input copy and step i-1's output copy
    run while step i computes.  Events order the three streams; the host
    never waits inside submit().
    """

    def __init__(self, layer: MoELayer, T: int, E: int, depth: int = 2, device="cuda"):
        dev = torch.device(device)
        self.layer, self.depth = layer, depth
        self.h2d = torch.cuda.Stream(device=dev)
        self.comp = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.bufs = [dict(logits=torch.empty(T, E, dtype=torch.float32, device=dev),
                          x=torch.empty(T, layer.H, dtype=torch.bfloat16, device=dev),
                          y=torch.empty(T, layer.H, dtype=torch.bfloat16, device=dev))
                     for _ in range(depth)]
        ev = lambda: [torch.cuda.Event() for _ in range(depth)]
        self.ev_in, self.ev_comp, self.ev_out = ev(), ev(), ev()
        self.used = [False] * depth
        self.i = 0

    def submit(self, logits_host: torch.Tensor, x_host: torch.Tensor, y_host: torch.Tensor):
        s = self.i % self.depth
        b = self.bufs[s]
        if self.used[s]:
            self.h2d.wait_event(self.ev_comp[s])     # the inputs' last reader is done
        with torch.cuda.stream(self.h2d):
            b["logits"].copy_(logits_host, non_blocking=True)
            b["x"].copy_(x_host, non_blocking=True)
        self.ev_in[s].record(self.h2d)
        self.comp.wait_event(self.ev_in[s])
        if self.used[s]:
            self.comp.wait_event(self.ev_out[s])     # the output's last copy is done
        self.layer.forward(b["logits"], b["x"], b["y"], self.comp)
        self.ev_comp[s].record(self.comp)
        self.d2h.wait_event(self.ev_comp[s])
        with torch.cuda.stream(self.d2h):
            y_host.copy_(b["y"], non_blocking=True)
        self.ev_out[s].record(self.d2h)
        self.used[s] = True
        self.i += 1

    def synchronize(self):
        for st in (self.h2d, self.comp, self.d2h):
            st.synchronize()
