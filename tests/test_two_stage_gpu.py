"""The two-stage comparator (pack into per-source send buffers laid out
[destination rank][local expert], then a separate all-to-all-v copy) against
the oracle: it must produce exactly the fused dispatch's receive rows,
metadata and inverse permutation ("[Infra-10] All-to-All Optimization", 4.3
and 5.2)."""
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
def test_two_stage_parity(gpu, name):
    wl = CASES[name]
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, two_stage=True)
    o = run_oracle(wl, inp)
    compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0


def test_two_stage_send_buffer_layout(gpu):
    """The send pool: source s's rows, destination ranks in order, each
    bucketed by local expert, (token, slot) order inside."""
    import torch
    wl = W.DECODE.scaled("decode_send", Tr=16, H=64)
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, two_stage=True)
    layer = g["layer"]
    send = layer.send_x.view(torch.int16).cpu().numpy().view(np.uint16)
    ids = g["ids"].reshape(-1)
    row = 0
    for s in range(wl.P):
        for e in range(wl.E):
            for a in range(s * wl.Tr * wl.k, (s + 1) * wl.Tr * wl.k):
                if ids[a] == e:
                    assert np.array_equal(send[row], inp.x[a // wl.k])
                    row += 1
    assert row == wl.Na
