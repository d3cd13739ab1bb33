"""The pplx-style fixed-slot comparator ("Efficient and portable MoE
communication", "Dispatch" / "Combine": private receive storage per source,
sized by the maximum tokens per rank) against the oracle.

The fixed-slot row of assignment (s, t, j) -> e is (e*P + s)*T_r + q, q its
rank among source s's assignments to e in (t, j) order. The oracle's compact
layout gives q as its receive row minus recv_offset[s][e], so every expected
row below is derived from the oracle alone. Payload, FP8 codes and scales,
metadata and the expert output at those rows, and the combined output, must
match the oracle exactly (route weights within 1 fp32 ulp)."""
import numpy as np
import pytest

import oracle
from combine_top_histogram_gb300 import workloads as W
from harness import bf16_ulp_diff, f32_ulp_diff, run_oracle, to_np_bits

pytestmark = pytest.mark.gpu

CASES = {
    "worked": W.WORKED,
    "decode_r": W.DECODE.scaled("fs_decode_r", Tr=37),
    "uniform_fp8_r": W.UNIFORM_FP8.scaled("fs_uniform_r", Tr=300, H=1024),
    "skewed_r": W.SKEWED.scaled("fs_skewed_r", Tr=700, H=512),
    "decode_full": W.DECODE,
}


def expected_rows(wl, o):
    lay = o["layout"]
    P, Tr, E, k = wl.P, wl.Tr, wl.E, wl.k
    inv_c = lay["inv"].reshape(-1).astype(np.int64)
    a = np.arange(wl.Na)
    s = a // (Tr * k)
    e = np.asarray(o["ids"]).reshape(-1).astype(np.int64)
    valid = inv_c >= 0
    q = inv_c - lay["recv_offset"].reshape(P, E)[s, np.where(valid, e, 0)]
    return np.where(valid, (e * P + s) * Tr + q, -1), inv_c


@pytest.mark.parametrize("name", list(CASES))
def test_fixed_slot_parity(gpu, name):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl = CASES[name]
    inp = W.make_inputs(wl)
    dev = torch.device("cuda")
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    c = torch.from_numpy(inp.expert_scale).to(dev) if inp.expert_scale is not None else None
    routed = inp.logits is not None
    if routed:
        layer.forward(x, logits=torch.from_numpy(inp.logits).to(dev), expert_scale=c,
                      fixed_slots=True)
    else:
        layer.forward(x, ids=torch.from_numpy(inp.ids).to(dev), w=torch.from_numpy(inp.w).to(dev),
                      expert_scale=c, fixed_slots=True)
    torch.cuda.synchronize()
    o = run_oracle(wl, inp)
    want, inv_c = expected_rows(wl, o)
    view = layer.layout_view()
    got_inv = view["inv"].cpu().numpy().astype(np.int64)
    assert np.array_equal(got_inv, want)
    assert layer.status() == 0
    # rows of each (expert, source) region: exactly cnt[s][e], packed from the region start
    rows = want[want >= 0]
    assert np.unique(rows).size == rows.size
    cnt = o["layout"]["cnt"].reshape(wl.P, wl.E)
    reg = rows // wl.Tr  # region index e*P + s
    fill = np.bincount(reg, minlength=wl.E * wl.P).reshape(wl.E, wl.P)
    assert np.array_equal(fill, cnt.T)
    assert np.all(rows % wl.Tr < cnt.T.reshape(-1)[reg])
    # payload, scales, metadata and expert output at the slot rows
    valid = want >= 0
    sel = torch.from_numpy(want[valid]).to(dev)
    src = inv_c[valid]
    s = layer.slots
    assert np.array_equal(to_np_bits(s["x"].index_select(0, sel)), o["recv_x"][src])
    if wl.dispatch_dtype == W.MOE_FP8_E4M3:
        assert np.array_equal(to_np_bits(s["scale"].index_select(0, sel)).view(np.uint32),
                              o["recv_scale"][src].view(np.uint32))
    for name_m in ("local_expert", "src_rank", "src_token", "slot"):
        assert np.array_equal(to_np_bits(s["meta"][name_m].index_select(0, sel)),
                              o["meta"][name_m][src]), name_m
    gw = to_np_bits(s["meta"]["weight"].index_select(0, sel))
    assert f32_ulp_diff(gw, o["meta"]["weight"][src]).max() <= (1 if routed else 0)
    assert np.array_equal(to_np_bits(s["y"].index_select(0, sel)), o["y"][src])
    assert bf16_ulp_diff(to_np_bits(layer.out), o["out"]).max() <= 1


def test_fixed_slots_refuse_a_capacity(gpu):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    wl = W.PREFILL.scaled("fs_cap", Tr=20, H=128, cap=30)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    layer.layout(torch.zeros((wl.T, wl.k), dtype=torch.int32, device="cuda"))
    x = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        layer.dispatch_fixed_slots(x, layer.w)
    meta = {n: torch.zeros(1, dtype=torch.int32, device="cuda")
            for n in ("local_expert", "src_rank", "src_token", "slot", "weight")}
    one = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_dispatch_fixed_slots(layer.handle, x, layer.w, one, one, meta)
    assert ei.value.code == -2


def test_fixed_slots_overflow_with_repeated_ids(gpu):
    """A region holds T_r rows: enough for distinct ids per token, not when an
    id repeats within a token. The excess of a (source, expert) pair is not
    written (inv = -1) and the status reports it; every other assignment lands
    at its slot row with the oracle's payload."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    P, Tr, E, k, H = 2, 5, 4, 3, 128
    wl = W.Workload("fs_overflow", P, Tr, E, k, H, W.MOE_BF16, "uniform", "identity")
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, (wl.T, k)).astype(np.int32)
    ids[:Tr] = 1  # source 0: every slot of every token picks expert 1 (15 > T_r = 5)
    w = rng.random((wl.T, k)).astype(np.float32)
    x = W.draw_hidden(rng, wl.T, H)
    inp = W.Inputs(wl, x, None, ids, w, None)
    o = run_oracle(wl, inp)
    want, inv_c = expected_rows(wl, o)
    q = np.where(want >= 0, want % Tr, 0)
    region_q = inv_c - o["layout"]["recv_offset"].reshape(P, E)[np.arange(wl.Na) // (Tr * k), ids.reshape(-1)]
    over = (inv_c >= 0) & (region_q >= Tr)
    assert over.sum() >= 10  # source 0: 15 assignments to expert 1, 5 fit
    want = np.where(over, -1, want)
    layer = MoeLayer(P, Tr, E, k, H)
    dev = torch.device("cuda")
    xt = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    layer.layout(torch.from_numpy(ids).to(dev))
    layer.dispatch_fixed_slots(xt, torch.from_numpy(w).to(dev))
    torch.cuda.synchronize()
    assert layer.status() & B.MOE_STATUS_SLOT_OVERFLOW
    got = layer.layout_view()["inv"].cpu().numpy().astype(np.int64)
    assert np.array_equal(got, want)
    ok = want >= 0
    sel = torch.from_numpy(want[ok]).to(dev)
    assert np.array_equal(to_np_bits(layer.slots["x"].index_select(0, sel)), o["recv_x"][inv_c[ok]])
    assert np.all(q[ok] < Tr)
