"""One MoE layer's dispatch/combine buffers and calls, over the C ABI.

``MoeLayer`` allocates (with torch) the workspace and the receive, metadata
and output buffers sized by the library's worst-case rule, then runs the path
through the binding: route+layout (or layout from given ids) -> dispatch ->
expert stand-in -> combine. Convenience for tests, the benchmark and smoke
checks; every step runs in the library's kernels.
"""
from __future__ import annotations

from . import binding as B


class MoeLayer:
    def __init__(self, P: int, Tr: int, E: int, k: int, H: int, dispatch_dtype: int = B.MOE_BF16,
                 cap: int = 0, device: str = "cuda"):
        import torch
        self.P, self.Tr, self.E, self.k, self.H = P, Tr, E, k, H
        self.T = P * Tr
        self.fp8 = dispatch_dtype == B.MOE_FP8_E4M3
        self.cfg = B.make_config(P, Tr, E, k, H, dispatch_dtype, cap)
        self.handle = B.moe_handle_create(self.cfg, device=device)
        self.rows = B.moe_recv_rows_max(self.cfg)
        dev = torch.device(device)
        rows, T = self.rows, self.T
        if self.fp8:
            self.recv_x = torch.empty((rows, H), dtype=torch.uint8, device=dev)
            self.recv_scale = torch.empty((rows, H // 128), dtype=torch.float32, device=dev)
        else:
            self.recv_x = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
            self.recv_scale = None
        self.meta = {
            "local_expert": torch.empty(rows, dtype=torch.int32, device=dev),
            "src_rank": torch.empty(rows, dtype=torch.int32, device=dev),
            "src_token": torch.empty(rows, dtype=torch.int32, device=dev),
            "slot": torch.empty(rows, dtype=torch.int32, device=dev),
            "weight": torch.empty(rows, dtype=torch.float32, device=dev),
        }
        self.y = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.slots = None  # fixed-slot buffers, allocated on first use
        self.fixed = False  # the last dispatch wrote the fixed-slot layout

    # -- steps ---------------------------------------------------------------
    def route_layout(self, logits, stream=None):
        """Fused top-k + count + scan; fills self.ids and self.w."""
        B.moe_route_dispatch_layout(self.handle, logits, self.ids, self.w, stream)

    def layout(self, ids, stream=None):
        B.moe_dispatch_layout(self.handle, ids, stream)

    def layout_tables(self, stream=None):
        """Per-source tables of the last layout without dispatching (a dispatch
        builds them in its own launch)."""
        B.moe_layout_tables(self.handle, stream)

    def dispatch(self, x, w, stream=None):
        B.moe_dispatch(self.handle, x, w, self.recv_x, self.recv_scale, self.meta, stream)
        self.fixed = False

    def dispatch_fixed_slots(self, x, w, stream=None):
        """The fixed-slot comparator: one region of T_r rows per (expert, source)
        (E*T rows in all); expert() and combine() then use these buffers."""
        import torch
        if self.slots is None:
            rows = B.moe_fixed_slot_rows(self.cfg)
            if rows == 0:
                raise ValueError("fixed slots need a configuration without capacity")
            dev = self.out.device
            sx = torch.empty((rows, self.H), dtype=torch.uint8 if self.fp8 else torch.bfloat16,
                             device=dev)
            self.slots = {
                "x": sx,
                "scale": (torch.empty((rows, self.H // 128), dtype=torch.float32, device=dev)
                          if self.fp8 else None),
                "meta": {n: torch.empty(rows, dtype=torch.float32 if n == "weight" else torch.int32,
                                        device=dev)
                         for n in ("local_expert", "src_rank", "src_token", "slot", "weight")},
                "y": torch.empty((rows, self.H), dtype=torch.bfloat16, device=dev),
            }
        s = self.slots
        B.moe_dispatch_fixed_slots(self.handle, x, w, s["x"], s["scale"], s["meta"], stream)
        self.fixed = True

    def dispatch_two_stage(self, x, w, stream=None):
        """The two-stage comparator: pack into per-source send buffers, then a
        separate all-to-all-v copy into the same receive layout."""
        import torch
        if getattr(self, "send_x", None) is None:
            self.send_x = torch.empty_like(self.recv_x)
            self.send_scale = (torch.empty_like(self.recv_scale)
                               if self.recv_scale is not None else None)
        B.moe_dispatch_two_stage(self.handle, x, w, self.send_x, self.send_scale, self.recv_x,
                                 self.recv_scale, self.meta, stream)
        self.fixed = False

    def dispatch_allgather(self, x, w, stream=None):
        """The AllGather comparator: all tokens to every rank, then a local filter."""
        import torch
        if getattr(self, "gathered_x", None) is None:
            dt = torch.uint8 if self.fp8 else torch.bfloat16
            self.gathered_x = torch.empty((self.P * self.T, self.H), dtype=dt,
                                          device=self.out.device)
            self.gathered_scale = (torch.empty((self.P * self.T, self.H // 128),
                                               dtype=torch.float32, device=self.out.device)
                                   if self.fp8 else None)
        B.moe_dispatch_allgather(self.handle, x, w, self.gathered_x, self.gathered_scale,
                                 self.recv_x, self.recv_scale, self.meta, stream)
        self.fixed = False

    def layout_dispatch_fused(self, x, ids=None, w=None, logits=None, stream=None):
        """One persistent launch: route (logits) or take ids/w, lay out, dispatch."""
        if logits is not None:
            ids, w = self.ids, self.w
        B.moe_layout_dispatch_fused(self.handle, logits, ids, w, x, self.recv_x, self.recv_scale,
                                    self.meta, stream)
        self.fixed = False

    def expert(self, expert_scale=None, stream=None):
        if self.fixed:
            s = self.slots
            B.moe_expert_standin(self.handle, s["x"], s["scale"], expert_scale, s["y"], stream)
            return
        B.moe_expert_standin(self.handle, self.recv_x, self.recv_scale, expert_scale, self.y,
                             stream)

    def combine(self, w, stream=None):
        B.moe_combine(self.handle, self.slots["y"] if self.fixed else self.y, w, self.out, stream)

    def forward(self, x, ids=None, w=None, logits=None, expert_scale=None, stream=None,
                two_stage=False, fused=False, allgather=False, fixed_slots=False):
        """Whole layer; with logits the routed ids/weights land in self.ids / self.w.
        two_stage=True dispatches through the two-stage comparator."""
        if fused:
            self.layout_dispatch_fused(x, ids, w, logits, stream)
            if logits is not None:
                w = self.w
            self.expert(expert_scale, stream)
            self.combine(w, stream)
            return self.out
        if logits is not None:
            self.route_layout(logits, stream)
            w = self.w
        else:
            self.layout(ids, stream)
        if allgather:
            self.dispatch_allgather(x, w, stream)
        elif fixed_slots:
            self.dispatch_fixed_slots(x, w, stream)
        elif two_stage:
            self.dispatch_two_stage(x, w, stream)
        else:
            self.dispatch(x, w, stream)
        self.expert(expert_scale, stream)
        self.combine(w, stream)
        return self.out

    def forward_pipelined(self, x, ids=None, w=None, logits=None, expert_scale=None, chunks=4,
                          stream=None):
        """The layer in token chunks on two streams: after the layout, chunk c+1's
        dispatch (main stream) overlaps chunk c's expert and combine (side
        stream, ordered after chunk c's dispatch by an event)."""
        import torch
        main = stream if stream is not None else torch.cuda.current_stream()
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(device=self.out.device)
        side = self._side
        self.fixed = False
        if logits is not None:
            self.route_layout(logits, main)
            w = self.w
        else:
            self.layout(ids, main)
        side.wait_stream(main)
        bounds = [self.T * c // chunks for c in range(chunks + 1)]
        for c in range(chunks):
            b0, b1 = bounds[c], bounds[c + 1]
            B.moe_dispatch_tokens(self.handle, b0, b1, x, w, self.recv_x, self.recv_scale,
                                  self.meta, main)
            ev = torch.cuda.Event()
            ev.record(main)
            side.wait_event(ev)
            B.moe_expert_standin_tokens(self.handle, b0, b1, self.recv_x, self.recv_scale,
                                        expert_scale, self.y, side)
            B.moe_combine_tokens(self.handle, b0, b1, self.y, w, self.out, side)
        main.wait_stream(side)
        return self.out

    def buffers(self) -> dict:
        """Every row buffer this layer owns, by name (those of the comparators
        only once they have been allocated by a first use)."""
        out = {"recv_x": self.recv_x, "y": self.y, "out": self.out}
        if self.recv_scale is not None:
            out["recv_scale"] = self.recv_scale
        out.update({"meta." + k: v for k, v in self.meta.items()})
        if getattr(self, "send_x", None) is not None:
            out["send_x"] = self.send_x
            if self.send_scale is not None:
                out["send_scale"] = self.send_scale
        if getattr(self, "gathered_x", None) is not None:
            out["gathered_x"] = self.gathered_x
            if self.gathered_scale is not None:
                out["gathered_scale"] = self.gathered_scale
        if self.slots is not None:
            out["slots.x"] = self.slots["x"]
            out["slots.y"] = self.slots["y"]
            if self.slots["scale"] is not None:
                out["slots.scale"] = self.slots["scale"]
            out.update({"slots.meta." + k: v for k, v in self.slots["meta"].items()})
        return out

    def poison(self, byte: int = 0xFF) -> None:
        """Fills every row buffer with one byte value (tests: rows a kernel must
        not write keep it, rows it must write lose it)."""
        import torch
        for t in self.buffers().values():
            t.view(-1).view(torch.uint8).fill_(byte)

    def layout_view(self) -> dict:
        return B.moe_get_layout(self.handle)

    def status(self, stream=None) -> int:
        return B.moe_read_status(self.handle, stream)

    def close(self):
        self.handle.close()
