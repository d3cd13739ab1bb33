"""The whole layer (route + layout, dispatch, expert stand-in, combine) captured
once in a CUDA graph and replayed with new inputs copied into the captured
tensors. Every call is asynchronous and keeps no per-call host state that a
replay would freeze, so each replay must match the oracle for its own inputs."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import bf16_ulp_diff, f32_ulp_diff, run_oracle, to_np_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("base", ["decode", "uniform_fp8"])
def test_layer_graph_replay(gpu, base):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl = {"decode": W.DECODE.scaled("graph_decode", Tr=37),
          "uniform_fp8": W.UNIFORM_FP8.scaled("graph_uniform", Tr=300, H=1024)}[base]
    dev = torch.device("cuda")
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    first = W.make_inputs(wl, seed=1)
    routed = first.logits is not None
    x = torch.from_numpy(first.x.view(np.int16)).to(dev).view(torch.bfloat16)
    z = torch.from_numpy(first.logits).to(dev) if routed else None
    ids = None if routed else torch.from_numpy(first.ids).to(dev)
    w = None if routed else torch.from_numpy(first.w).to(dev)
    c = torch.from_numpy(first.expert_scale).to(dev) if first.expert_scale is not None else None

    def layer_call():
        if routed:
            layer.forward(x, logits=z, expert_scale=c)
        else:
            layer.forward(x, ids=ids, w=w, expert_scale=c)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer_call()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer_call()
    for seed in (2, 3, 4):
        inp = W.make_inputs(wl, seed=seed)
        x.copy_(torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16))
        if routed:
            z.copy_(torch.from_numpy(inp.logits).to(dev))
        else:
            ids.copy_(torch.from_numpy(inp.ids).to(dev))
            w.copy_(torch.from_numpy(inp.w).to(dev))
        if c is not None:
            c.copy_(torch.from_numpy(inp.expert_scale).to(dev))
        graph.replay()
        torch.cuda.synchronize()
        o = run_oracle(wl, inp)
        if routed:
            assert np.array_equal(layer.ids.cpu().numpy(), o["ids"]), seed
            assert f32_ulp_diff(layer.w.cpu().numpy(), o["w"]).max() <= 1, seed
        view = layer.layout_view()
        assert np.array_equal(view["inv"].cpu().numpy(), o["layout"]["inv"].reshape(-1)), seed
        assert np.array_equal(view["expert_offset"].cpu().numpy(), o["layout"]["expert_offset"]), seed
        assert bf16_ulp_diff(to_np_bits(layer.out), o["out"]).max() <= 1, seed
    assert layer.status() == 0
