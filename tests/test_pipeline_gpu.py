"""The token-chunked dispatch -> expert -> combine pipeline on two streams
("[Infra-10] All-to-All Optimization", 7: start the expert as soon as its
inputs arrive; "Expert Parallel: MoE Token ...", overlap section) against the
oracle: any chunking must give exactly the whole-layer result."""
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("decode_r", W.DECODE.scaled("decode_r", Tr=37), 3),
    ("decode_full", W.DECODE, 4),
    ("uniform_fp8_r", W.UNIFORM_FP8.scaled("uniform_fp8_r", Tr=300), 5),
    ("skewed_r", W.SKEWED.scaled("skewed_r", Tr=700), 2),
    ("prefill_r_cap", W.PREFILL.scaled("prefill_r", Tr=60, cap=50), 7),
    ("one_chunk", W.WORKED, 1),
    ("more_chunks_than_tokens", W.WORKED, 11),
]


@pytest.mark.parametrize("name,wl,chunks", CASES, ids=[c[0] for c in CASES])
def test_pipelined_parity(gpu, name, wl, chunks):
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, pipelined=chunks)
    o = run_oracle(wl, inp)
    compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0


def test_token_range_arguments_are_checked(gpu):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    wl = W.WORKED
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H)
    x = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((wl.T, wl.k), dtype=torch.float32, device="cuda")
    ids = torch.zeros((wl.T, wl.k), dtype=torch.int32, device="cuda")
    layer.layout(ids)
    for b0, b1 in [(-1, 2), (3, 2), (0, wl.T + 1)]:
        with pytest.raises(B.MoeError):
            B.moe_dispatch_tokens(layer.handle, b0, b1, x, w, layer.recv_x, None, layer.meta)
