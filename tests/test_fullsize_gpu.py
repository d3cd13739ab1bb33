"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (one MoeLayer per workload: fused route+layout or layout,
dispatch, expert stand-in, combine). Decode, uniform-FP8 and skewed are
compared element by element against the oracle; prefill (1,048,576
assignments, 27 GB of buffers) compares the whole layout and permutation, and
the payload, scales, metadata and combined rows of sampled tokens, each
recomputed by the oracle from that token's inputs alone."""
import numpy as np
import pytest

import oracle
from combine_top_histogram_gb300 import workloads as W
from harness import (LAYOUT_KEYS, bf16_ulp_diff, compare, f32_ulp_diff, run_gpu, run_oracle,
                     to_np_bits)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["worked", "decode", "uniform_fp8", "skewed"])
def test_full_size_parity(gpu, name):
    wl = W.CONFIGS[name]
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp)
    o = run_oracle(wl, inp)
    st = compare(wl, g, o, routed=inp.logits is not None)
    assert g["status"] == 0
    assert st["kept"] == wl.Na


def test_prefill_full_width_staged_fp8_dispatch_every_element(gpu):
    """The kernel full-size prefill times: at H = 7168 with at least 16 tokens
    per dispatch CTA the FP8 dispatch stages each CTA's next token row in
    shared memory (four 16-value chunks per thread). Prefill's per-token
    distribution, capacity rule and expert stand-in at 32 x 1300 tokens
    (332,800 assignments): every receive row, scale, metadata element, expert
    row and combined row against the oracle."""
    import os

    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Tr = 1300
    wl = W.PREFILL.scaled("prefill_tr1300", Tr=Tr, cap=W.prefill_capacity(32 * Tr, 8, 256))
    # the launch takes min(T, 16 * SMs) CTAs and stages rows from 16 tokens per CTA
    assert wl.T >= 16 * 16 * sms and wl.H // 16 > 256
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp)
    o = run_oracle(wl, inp, threads=os.cpu_count() or 1)
    st = compare(wl, g, o, routed=True)
    assert g["status"] == 0
    assert st["kept"] == int(o["layout"]["totals"][0]) > 0.99 * wl.Na


def test_full_size_prefill_sampled(gpu):
    import torch
    wl = W.PREFILL
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, copy_rows=False)
    layer = g["layer"]
    assert g["status"] == 0
    # route: ids exact and weights within 1 ulp for every token
    ids, w = oracle.route_topk(inp.logits, wl.k)
    assert np.array_equal(g["ids"], ids)
    assert f32_ulp_diff(g["w"], w).max() <= 1
    # whole layout and permutation
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, ids, wl.cap)
    for gk, ok in LAYOUT_KEYS:
        assert np.array_equal(g[gk].reshape(-1), lay[ok].reshape(-1)), gk
    assert g["totals"][:3].tolist() == lay["totals"].tolist()
    # sampled tokens: payload rows, scales, metadata and the combined row
    rng = np.random.default_rng(123)
    tokens = np.unique(np.concatenate([rng.integers(0, wl.T, 96), [0, wl.T - 1]]))
    inv = lay["inv"].reshape(wl.T, wl.k)

    def rows_of(t, idx):
        sel = torch.from_numpy(np.asarray(idx, np.int64)).to(t.device)
        return to_np_bits(t.index_select(0, sel))

    for gtok in tokens:
        q, sc = oracle.quantize_row_fp8(inp.x[gtok])
        yrow = oracle.expert_dequant_fp8(q[None, :], sc[None, :])[0]
        rows = [int(r) for r in inv[gtok] if r >= 0]
        slots = [j for j in range(wl.k) if inv[gtok, j] >= 0]
        if rows:
            rx, rs, ry = (rows_of(layer.recv_x, rows), rows_of(layer.recv_scale, rows),
                          rows_of(layer.y, rows))
            meta = {k: rows_of(v, rows) for k, v in layer.meta.items()}
            for i, (r, j) in enumerate(zip(rows, slots)):
                assert np.array_equal(rx[i], q)
                assert np.array_equal(rs[i].view(np.uint32), sc.view(np.uint32))
                assert meta["src_rank"][i] == gtok // wl.Tr
                assert meta["src_token"][i] == gtok % wl.Tr
                assert meta["slot"][i] == j
                assert meta["local_expert"][i] == ids[gtok, j] % wl.L
                assert f32_ulp_diff(meta["weight"][i:i + 1], w[gtok, j:j + 1]).max() <= 1
                assert np.array_equal(ry[i], yrow)
        # the token's k rows are all the dequantised token row; local inv
        local_inv = np.where(inv[gtok] >= 0, np.arange(wl.k), -1).astype(np.int32)
        want = oracle.combine_token(local_inv, w[gtok], np.repeat(yrow[None, :], wl.k, 0))
        got = rows_of(layer.out, [gtok])[0]
        assert bf16_ulp_diff(got, want).max() <= 1
