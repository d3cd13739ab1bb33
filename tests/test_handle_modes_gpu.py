"""One handle through every dispatch mode in turn: separate, persistent,
fixed slots, two-stage, AllGather, pipelined, separate again. Each layer has
its own routing (a new seed) and must match the oracle exactly, so the
handle's state carried between calls (the per-expert totals cleared by each
scan, the per-source tables built by whichever dispatch comes first, the
slot-row flag of the expert stand-in) is exercised across every transition."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import bf16_ulp_diff, compare, run_gpu, run_oracle, to_np_bits
from test_fixed_slots_gpu import expected_rows

pytestmark = pytest.mark.gpu

MODES = ["separate", "fused", "fixed_slots", "two_stage", "allgather", "pipelined", "separate"]


@pytest.mark.parametrize("base", ["decode", "uniform_fp8"])
def test_one_handle_through_every_mode(gpu, base):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl = {"decode": W.DECODE.scaled("modes_decode", Tr=37),
          "uniform_fp8": W.UNIFORM_FP8.scaled("modes_uniform", Tr=300, H=1024)}[base]
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    dev = torch.device("cuda")
    for i, mode in enumerate(MODES):
        inp = W.make_inputs(wl, seed=100 + i)
        o = run_oracle(wl, inp)
        routed = inp.logits is not None
        if mode == "fixed_slots":
            x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
            c = torch.from_numpy(inp.expert_scale).to(dev) if inp.expert_scale is not None else None
            if routed:
                layer.forward(x, logits=torch.from_numpy(inp.logits).to(dev), expert_scale=c,
                              fixed_slots=True)
            else:
                layer.forward(x, ids=torch.from_numpy(inp.ids).to(dev),
                              w=torch.from_numpy(inp.w).to(dev), expert_scale=c, fixed_slots=True)
            torch.cuda.synchronize()
            want, _ = expected_rows(wl, o)
            got = layer.layout_view()["inv"].cpu().numpy().astype(np.int64)
            assert np.array_equal(got, want), (i, mode)
            assert bf16_ulp_diff(to_np_bits(layer.out), o["out"]).max() <= 1, (i, mode)
            assert layer.status() == 0
            continue
        g = run_gpu(wl, inp, layer=layer, fused=mode == "fused", two_stage=mode == "two_stage",
                    allgather=mode == "allgather", pipelined=4 if mode == "pipelined" else 0)
        compare(wl, g, o, routed=routed)
        assert g["status"] == 0, (i, mode)


def _inputs_to_device(inp, dev):
    import torch
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    z = torch.from_numpy(inp.logits).to(dev) if inp.logits is not None else None
    ids = torch.from_numpy(inp.ids).to(dev) if inp.ids is not None else None
    w = torch.from_numpy(inp.w).to(dev) if inp.w is not None else None
    c = torch.from_numpy(inp.expert_scale).to(dev) if inp.expert_scale is not None else None
    return x, z, ids, w, c


def _check_layer(layer, wl, inp):
    o = run_oracle(wl, inp)
    view = layer.layout_view()
    assert np.array_equal(view["inv"].cpu().numpy(), o["layout"]["inv"].reshape(-1))
    assert bf16_ulp_diff(to_np_bits(layer.out), o["out"]).max() <= 1
    assert layer.status() == 0


def test_two_handles_interleaved_and_on_two_streams(gpu):
    """Two handles share no state: their calls interleaved on one stream, then
    two whole layers on two concurrent streams, each exact."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    dev = torch.device("cuda")
    wa = W.DECODE.scaled("pair_a", Tr=37)
    wb = W.UNIFORM_FP8.scaled("pair_b", Tr=300, H=1024)
    la = MoeLayer(wa.P, wa.Tr, wa.E, wa.k, wa.H, wa.dispatch_dtype, wa.cap)
    lb = MoeLayer(wb.P, wb.Tr, wb.E, wb.k, wb.H, wb.dispatch_dtype, wb.cap)
    ia, ib = W.make_inputs(wa, seed=7), W.make_inputs(wb, seed=8)
    xa, za, _, _, ca = _inputs_to_device(ia, dev)
    xb, _, idsb, wbt, cb = _inputs_to_device(ib, dev)
    # interleaved on the current stream
    la.route_layout(za)
    lb.layout(idsb)
    la.dispatch(xa, la.w)
    lb.dispatch(xb, wbt)
    lb.expert(cb)
    la.expert(ca)
    la.combine(la.w)
    lb.combine(wbt)
    torch.cuda.synchronize()
    _check_layer(la, wa, ia)
    _check_layer(lb, wb, ib)
    # concurrently on two streams, new routings
    ia, ib = W.make_inputs(wa, seed=9), W.make_inputs(wb, seed=10)
    xa, za, _, _, ca = _inputs_to_device(ia, dev)
    xb, _, idsb, wbt, cb = _inputs_to_device(ib, dev)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    la.forward(xa, logits=za, expert_scale=ca, stream=sa)
    lb.forward(xb, ids=idsb, w=wbt, expert_scale=cb, stream=sb)
    torch.cuda.synchronize()
    _check_layer(la, wa, ia)
    _check_layer(lb, wb, ib)
