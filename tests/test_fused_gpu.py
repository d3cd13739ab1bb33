"""The persistent single-launch path (route/count/scan/dispatch in one
cooperative kernel with bounded grid barriers) against the oracle, and its
timeout path: a wait limit of zero makes every grid barrier give up at once,
which must set MOE_STATUS_TIMEOUT and return, leaving the next call exact.
("[Infra-10] All-to-All Optimization", 9-10: persistent kernels and device-side
synchronisation for the low-latency decode mode.)"""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    "worked": W.WORKED,
    "decode_r": W.DECODE.scaled("decode_r", Tr=37),
    "decode_full": W.DECODE,
    "uniform_fp8_r": W.UNIFORM_FP8.scaled("uniform_fp8_r", Tr=1100),
    "skewed_r": W.SKEWED.scaled("skewed_r", Tr=2500),
    # 25 tokens x 14 KB per chunk exceed the shared-memory staging: direct loads
    "prefill_r_cap": W.PREFILL.scaled("prefill_r", Tr=100, cap=90),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_parity(gpu, name):
    wl = CASES[name]
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, fused=True)
    o = run_oracle(wl, inp)
    compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0


def test_fused_with_padding_and_invalid_ids(gpu):
    rng = np.random.default_rng(21)
    wl = W.Workload("fused_pad", 4, 60, 16, 3, 256, W.MOE_BF16, "uniform", "identity", cap=20)
    x = W.draw_hidden(rng, wl.T, wl.H)
    ids = np.stack([rng.permutation(wl.E)[:wl.k] for _ in range(wl.T)]).astype(np.int32)
    ids = W.mask_random_slots(ids, 0.2, 3)
    ids[5, 1] = 77  # out of range: masked and flagged
    w = rng.random((wl.T, wl.k)).astype(np.float32)
    inp = W.Inputs(wl, x, None, ids, w, None)
    g = run_gpu(wl, inp, fused=True)
    from combine_top_histogram_gb300.binding import MOE_STATUS_BAD_EXPERT_ID
    assert g["status"] == MOE_STATUS_BAD_EXPERT_ID
    compare(wl, g, run_oracle(wl, inp), routed=False)


def test_fused_rejects_chunks_beyond_its_limit(gpu):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    wl = W.PREFILL  # 1024 tokens x top-8 per chunk > 4096 assignments
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, 128, wl.dispatch_dtype, wl.cap)
    x = torch.zeros((wl.T, 128), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((wl.T, wl.E), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        layer.layout_dispatch_fused(x, logits=z)
    assert ei.value.code == -2


def test_fused_grid_barrier_timeout_is_reported_and_recoverable(gpu):
    """The wait limit is injected from the host (0 polls): nothing is made to
    hang or fault. After the timed-out calls every slot's inv is -1 or a row in
    range, and a call with the normal limit is exact again."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    wl = W.DECODE.scaled("fused_timeout", Tr=64, H=256)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    inp = W.make_inputs(wl)
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    z = torch.from_numpy(inp.logits).cuda()
    B.moe_set_wait_limit(layer.handle, 0)
    for _ in range(3):
        layer.layout_dispatch_fused(x, logits=z)
        assert layer.status() & B.MOE_STATUS_TIMEOUT
        inv = layer.layout_view()["inv"].cpu().numpy()
        assert inv.min() >= -1 and inv.max() < layer.rows
    B.moe_set_wait_limit(layer.handle, 1 << 22)
    g = run_gpu(wl, inp, layer=layer, fused=True)
    assert g["status"] == 0
    compare(wl, g, run_oracle(wl, inp), routed=True)
