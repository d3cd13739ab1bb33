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
