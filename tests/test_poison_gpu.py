"""Poisoned buffers, in every dispatch mode: a stand-in for a memory checker
(compute-sanitizer is closed on this machine).

Every row buffer of a layer is filled with 0xFF bytes before the layer runs.
Afterwards the rows a kernel must write hold no 0xFF pattern (an e4m3 0xFF
code, a bf16 0xFFFF or an fp32/int32 of all ones is a NaN or -1 that a valid
row never holds), and every row it must not write still holds nothing else:
a stray write past the kept rows, or a row left unwritten, fails the test.
This checks what the pages warn about ("Expert Parallel: MoE Token ...",
"Correctness checks come before tuning": a wrong offset silently adds one
token's output to another's) beyond the oracle comparison of rows [0, kept).
"""
import numpy as np
import pytest

import oracle
from combine_top_histogram_gb300 import workloads as W
from harness import compare, run_gpu, run_oracle, to_np_bits

pytestmark = pytest.mark.gpu

MODES = ["separate", "fused", "two_stage", "allgather", "pipelined"]


def _bf16_given_ids():
    wl = W.SKEWED.scaled("poison_skewed", Tr=300, H=256)
    inp = W.make_inputs(wl)
    inp.ids = W.mask_random_slots(inp.ids, 0.1, 7)
    return wl, inp


def _fp8_routed_with_drops():
    wl = W.PREFILL.scaled("poison_prefill", Tr=40, H=256, cap=42)
    return wl, W.make_inputs(wl)


def _all_ff(a):
    b = np.ascontiguousarray(a).view(np.uint8)
    return bool((b == 0xFF).all())


def _any_poison_element(a):
    """Some element of a is the all-ones pattern of its own width."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint8:
        return bool((a == 0xFF).any())
    if a.dtype in (np.uint16, np.int16):
        return bool((a.view(np.uint16) == 0xFFFF).any())
    return bool((a.view(np.uint32) == 0xFFFFFFFF).any())


def _check_rows(name, arr, written_rows):
    """written_rows: boolean mask over the first axis."""
    assert not _any_poison_element(arr[written_rows]), f"{name}: a row to be written was not"
    assert _all_ff(arr[~written_rows]), f"{name}: a row outside the kept rows was written"


def _fp8_many_tokens_with_drops():
    """Over 16 tokens per dispatch CTA and H a multiple of 512: the receive
    rows are stored by bulk copies from shared memory."""
    wl = W.UNIFORM_FP8.scaled("poison_bulk", Tr=5000, H=512, cap=1200)
    return wl, W.make_inputs(wl)


CASES = {"bf16_given_ids": _bf16_given_ids, "fp8_routed_drops": _fp8_routed_with_drops,
         "fp8_bulk_drops": _fp8_many_tokens_with_drops}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", list(CASES))
def test_poisoned_buffers(gpu, mode, case):
    from combine_top_histogram_gb300 import MoeLayer
    wl, inp = CASES[case]()
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap, "cuda:0")
    flags = dict(two_stage=mode == "two_stage", fused=mode == "fused",
                 allgather=mode == "allgather", pipelined=3 if mode == "pipelined" else 0)
    run_gpu(wl, inp, layer=layer, copy_rows=False, **flags)  # allocates the mode's buffers
    layer.poison()
    g = run_gpu(wl, inp, layer=layer, **flags)
    o = run_oracle(wl, inp)
    st = compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0
    n = st["kept"]
    if case in ("fp8_routed_drops", "fp8_bulk_drops"):
        assert o["layout"]["totals"][1] > 0  # the capacity dropped rows
    if case == "bf16_given_ids":
        assert o["layout"]["totals"][2] > 0  # some slots were masked
    bufs = {k: to_np_bits(v) for k, v in layer.buffers().items()}
    kept = np.arange(layer.rows) < n
    for name, arr in bufs.items():
        if name in ("out", "gathered_x", "gathered_scale"):
            # every token's restored row; every gathered copy of every token
            assert not _any_poison_element(arr), f"{name}: a row was not written"
        else:
            _check_rows(name, arr, kept)


def test_poisoned_buffers_fixed_slots(gpu):
    """Fixed per-(source, expert) slots: region (e, s) holds exactly cnt[s][e]
    filled rows at its start; every other slot row keeps the poison."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl, inp = _bf16_given_ids()
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap, "cuda:0")
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(inp.ids).cuda()
    w = torch.from_numpy(inp.w).cuda()
    layer.forward(x, ids=ids, w=w, fixed_slots=True)
    layer.poison()
    layer.forward(x, ids=ids, w=w, fixed_slots=True)
    assert layer.status() == 0
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, inp.ids, 0)
    rows = layer.slots["x"].shape[0]
    filled = np.zeros(rows, bool)
    for s in range(wl.P):
        for e in range(wl.E):
            base = (e * wl.P + s) * wl.Tr
            filled[base:base + lay["cnt"][s, e]] = True
    for name, arr in layer.buffers().items():
        a = to_np_bits(arr)
        if name.startswith("slots."):
            _check_rows(name, a, filled)
        elif name == "out":
            assert not _any_poison_element(a)
        else:  # the compact buffers are not used by this mode
            assert _all_ff(a), name
    out_o = run_oracle(wl, inp)["out"]
    assert np.array_equal(to_np_bits(layer.out), out_o)
