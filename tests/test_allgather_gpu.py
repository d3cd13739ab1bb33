"""The AllGather-style dispatcher comparator ("Expert Parallel: MoE Token ...",
"Why not collect all tokens with AllGather": every rank gathers every token and
filters its own assignments) against the oracle: exactly the fused dispatch's
receive rows, metadata and inverse permutation."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    "worked": W.WORKED,
    "decode_r": W.DECODE.scaled("decode_r", Tr=37),
    "uniform_fp8_r": W.UNIFORM_FP8.scaled("uniform_fp8_r", Tr=300),
    "skewed_r": W.SKEWED.scaled("skewed_r", Tr=700),
    "prefill_r_cap": W.PREFILL.scaled("prefill_r", Tr=60, cap=50),
}


@pytest.mark.parametrize("name", list(CASES))
def test_allgather_parity(gpu, name):
    wl = CASES[name]
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, allgather=True)
    o = run_oracle(wl, inp)
    compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0


def test_allgather_copies_every_token_to_every_rank(gpu):
    import torch
    wl = W.DECODE.scaled("ag_copies", Tr=5, H=64)
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, allgather=True)
    gx = g["layer"].gathered_x.view(torch.int16).cpu().numpy().view(np.uint16)
    for d in range(wl.P):
        assert np.array_equal(gx[d * wl.T:(d + 1) * wl.T], inp.x)
