"""Byte accounting for the dispatch/combine path (measurement only).

Two views, kept apart as the pages ask ("Expert Parallel: MoE Token ...",
"What to record when evaluating EP": say whether a bandwidth is logical or
physical):

* wire payload -- what the all-to-all-v hops carry: rows x H x bytes per hop
  ("Expert Parallel ...", "Traffic should be estimated per assignment": one
  dispatch carries N_t*k*H*b, combine returns the same shape);
* algorithmic HBM bytes -- what each kernel must read and write at least once
  on one GPU (the roofline numerator): the token rows read once, the k
  payload rows written, scales and metadata, the k expert rows read back and
  the restored rows written.
"""
from __future__ import annotations

import dataclasses


def wire_payload_bytes(T: int, k: int, H: int, dispatch_bytes: float, combine_bytes: float) -> int:
    """Dispatch plus combine payload of one layer round trip, metadata excluded."""
    return int(T * k * H * dispatch_bytes + T * k * H * combine_bytes)


@dataclasses.dataclass(frozen=True)
class KernelBytes:
    layout: int
    dispatch: int
    combine: int

    @property
    def total(self) -> int:
        return self.layout + self.dispatch + self.combine


def hbm_bytes(P: int, Tr: int, E: int, k: int, H: int, fp8: bool, rows: int | None = None,
              routed: bool = False) -> KernelBytes:
    """Algorithmic HBM bytes per launch of each kernel.

    rows: kept receive rows (defaults to T*k, i.e. no drops, no padding).
    routed: the layout kernel reads logits and writes ids and weights.
    """
    T = P * Tr
    Na = T * k
    rows = Na if rows is None else rows
    elt = 1 if fp8 else 2
    # layout: ids (or logits + routed ids/weights) in, assignment codes out.
    layout = (T * E * 4 + Na * 8 if routed else Na * 4) + Na * 4
    # dispatch: x once, k payload rows (+ scales), 20 B of metadata per row,
    # the assignment code and weight of every slot, inv out.
    dispatch = T * H * 2 + rows * H * elt + (rows * (H // 128) * 4 if fp8 else 0) \
        + rows * 20 + Na * 4 + rows * 4 + Na * 4
    # combine: k expert rows in, inv + weights, one restored row out.
    combine = rows * H * 2 + Na * 8 + T * H * 2
    return KernelBytes(layout, dispatch, combine)


def payload_bytes(P: int, Tr: int, k: int, H: int, fp8: bool, rows: int | None = None) -> dict:
    """Token-row bytes only (the figures in the workload table): dispatch =
    x read + payload rows (+ scales) written; combine = rows read + out written."""
    T = P * Tr
    rows = T * k if rows is None else rows
    elt = 1 if fp8 else 2
    d = T * H * 2 + rows * H * elt + (rows * (H // 128) * 4 if fp8 else 0)
    c = rows * H * 2 + T * H * 2
    return {"dispatch": d, "combine": c, "total": d + c}
