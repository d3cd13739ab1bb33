"""Small layouts skip the scan kernel: the dispatch right after a layout lays
itself out from the totals the layout kernel accumulated (the direct
dispatch), and any other consumer of that layout scans first. These tests
drive one handle through the transitions: a layout that nothing consumes
followed by another, a direct dispatch followed by the scanned modes on the
same layout, the persistent path in between, and token-range dispatches,
each checked against the oracle."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import LAYOUT_KEYS, bf16_ulp_diff, compare, run_oracle, to_np_bits

pytestmark = pytest.mark.gpu


def _dev(inp):
    import torch
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    z = torch.from_numpy(inp.logits).cuda() if inp.logits is not None else None
    ids = torch.from_numpy(inp.ids).cuda() if inp.ids is not None else None
    w = torch.from_numpy(inp.w).cuda() if inp.w is not None else None
    c = torch.from_numpy(inp.expert_scale).cuda() if inp.expert_scale is not None else None
    return x, z, ids, w, c


def _result(layer, inp):
    import torch
    torch.cuda.synchronize()
    view = layer.layout_view()
    g = {k: to_np_bits(v) for k, v in view.items()}
    g["ids"] = to_np_bits(layer.ids) if inp.logits is not None else None
    g["w"] = to_np_bits(layer.w) if inp.logits is not None else inp.w
    g["recv_x"] = to_np_bits(layer.recv_x)
    g["recv_scale"] = to_np_bits(layer.recv_scale) if layer.recv_scale is not None else None
    g["meta"] = {k: to_np_bits(v) for k, v in layer.meta.items()}
    g["y"] = to_np_bits(layer.y)
    g["out"] = to_np_bits(layer.out)
    g["status"] = layer.status()
    return g


@pytest.mark.parametrize("base", ["decode", "uniform_fp8"])
def test_one_layout_through_direct_then_scanned_modes(gpu, base):
    from combine_top_histogram_gb300 import MoeLayer
    wl = {"decode": W.DECODE.scaled("direct_decode", Tr=37),
          "uniform_fp8": W.UNIFORM_FP8.scaled("direct_uniform", Tr=300, H=1024)}[base]
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    routed = wl.routing == "logits"
    # a layout that nothing consumes: its totals must not leak into the next
    junk = W.make_inputs(wl, seed=50)
    x, z, ids, w, c = _dev(junk)
    if routed:
        layer.route_layout(z)
    else:
        layer.layout(ids)
    inp = W.make_inputs(wl, seed=51)
    o = run_oracle(wl, inp)
    x, z, ids, w, c = _dev(inp)
    if routed:
        layer.route_layout(z)
        w = layer.w
    else:
        layer.layout(ids)
    # direct dispatch, then the other dispatch modes on the same layout
    for mode in ["direct", "two_stage", "allgather", "separate_again"]:
        layer.poison()
        if mode == "two_stage":
            layer.dispatch_two_stage(x, w)
        elif mode == "allgather":
            layer.dispatch_allgather(x, w)
        else:
            layer.dispatch(x, w)
        layer.expert(c)
        layer.combine(w)
        g = _result(layer, inp)
        compare(wl, g, o, routed=routed)
        assert g["status"] == 0, mode


def test_direct_and_scanned_layouts_alternate(gpu):
    """Layout + dispatch (direct), layout + token ranges (scanned), layout +
    tables only, persistent path, layout + dispatch again: every layer exact."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl = W.SKEWED.scaled("direct_alt", Tr=400, H=256)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    for i, mode in enumerate(["direct", "pipelined", "tables", "fused", "direct"]):
        inp = W.make_inputs(wl, seed=60 + i)
        inp.ids = W.mask_random_slots(inp.ids, 0.05, 60 + i)
        o = run_oracle(wl, inp)
        x, _, ids, w, c = _dev(inp)
        if mode == "pipelined":
            layer.forward_pipelined(x, ids=ids, w=w, expert_scale=c, chunks=3)
        elif mode == "fused":
            layer.forward(x, ids=ids, w=w, expert_scale=c, fused=True)
        elif mode == "tables":
            layer.layout(ids)
            layer.layout_tables()
            torch.cuda.synchronize()
            view = {k: to_np_bits(v) for k, v in layer.layout_view().items()}
            for gk, ok in LAYOUT_KEYS:
                if gk != "inv":
                    assert np.array_equal(view[gk].reshape(-1), o["layout"][ok].reshape(-1)), gk
            layer.dispatch(x, w)
            layer.expert(c)
            layer.combine(w)
        else:
            layer.forward(x, ids=ids, w=w, expert_scale=c)
        g = _result(layer, inp)
        compare(wl, g, o, routed=False)
        assert g["status"] == 0, mode
