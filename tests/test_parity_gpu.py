"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, on the five workloads at reduced sizes (several layout chunks, a
ragged last chunk, full row widths) and on the pages' edge cases ("Expert
Parallel: MoE Token ...", "Correctness checks come before tuning": all tokens
local, all to one remote rank, extreme skew, empty experts, token counts off
the alignment, top-1 / top-2 / larger k, padding, capacity and invalid tokens,
rank reordering)."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W
from harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _check(wl, inp=None, ids=None):
    inp = inp or W.make_inputs(wl)
    g = run_gpu(wl, inp, ids=ids)
    w = None
    if ids is not None and inp.w is None:
        raise ValueError("ids override needs weights")
    o = run_oracle(wl, inp, ids=ids, w=w)
    st = compare(wl, g, o, routed=(ids is None and inp.logits is not None))
    assert g["status"] == 0
    return g, o, st


REDUCED = {
    "worked": W.WORKED,
    "decode": W.DECODE.scaled("decode_r", Tr=37),
    "uniform_fp8": W.UNIFORM_FP8.scaled("uniform_fp8_r", Tr=1100),
    "skewed": W.SKEWED.scaled("skewed_r", Tr=2500),
    "prefill_cap_tight": W.PREFILL.scaled("prefill_r", Tr=100, cap=90),
    "prefill_cap_formula": W.PREFILL.scaled(
        "prefill_r2", Tr=100, cap=W.prefill_capacity(32 * 100, 8, 256)),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_workload_parity_reduced(gpu, name):
    wl = REDUCED[name]
    g, o, st = _check(wl)
    if name == "prefill_cap_tight":
        assert o["layout"]["totals"][1] > 0, "the tight capacity must drop rows"
    if name == "worked":
        # the printed receive lists, read from the GPU's metadata
        from golden_io import worked_example
        _, recv, _ = worked_example()
        eoff = g["expert_offset"]
        for (r, e), tokens in recv.items():
            rows = range(eoff[e], eoff[e + 1])
            got = [int(g["meta"]["src_rank"][i]) * 2 + int(g["meta"]["src_token"][i]) for i in rows]
            assert got == tokens


def _bf16_case(P, Tr, E, k, H, ids, cap=0, seed=0, w=None):
    wl = W.Workload(f"edge_{P}_{Tr}_{E}_{k}_{H}", P, Tr, E, k, H, W.MOE_BF16, "uniform",
                    "identity", cap=cap, seed=seed)
    rng = np.random.default_rng(seed)
    x = W.draw_hidden(rng, wl.T, H)
    if w is None:
        w = rng.random((wl.T, k)).astype(np.float32)
    inp = W.Inputs(wl, x, None, np.ascontiguousarray(ids, np.int32), w, None)
    return _check(wl, inp)


def test_edge_all_local(gpu):
    P, Tr, E, k = 4, 33, 8, 2
    ids = np.array([[2 * (g // Tr), 2 * (g // Tr) + 1] for g in range(P * Tr)])
    g, o, _ = _bf16_case(P, Tr, E, k, 256, ids)
    assert np.array_equal(g["count_matrix"], np.diag([Tr * k] * P))


def test_edge_all_to_one_remote_rank_and_empty_experts(gpu):
    P, Tr, E, k = 4, 45, 8, 2
    ids = np.tile([[7, 6]], (P * Tr, 1))
    g, o, _ = _bf16_case(P, Tr, E, k, 136, ids)
    assert g["count_matrix"][:, 3].tolist() == [Tr * k] * P
    assert g["expert_count"][:6].sum() == 0


def test_edge_extreme_skew_with_capacity(gpu):
    rng = np.random.default_rng(3)
    P, Tr, E, k = 8, 300, 16, 2
    ids = np.stack([[0, 1 + rng.integers(0, 15)] for _ in range(P * Tr)])
    g, o, st = _bf16_case(P, Tr, E, k, 64, ids, cap=500)
    assert g["totals"][1] == P * Tr - 500  # expert 0 overflows


def test_edge_padding_and_invalid_ids(gpu):
    rng = np.random.default_rng(4)
    P, Tr, E, k = 2, 77, 6, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)]).astype(np.int32)
    ids = W.mask_random_slots(ids, 0.3, 5)
    ids[:5, 0] = -1  # all-masked tokens combine to zero
    ids[:5, 1:] = -1
    g, o, _ = _bf16_case(P, Tr, E, k, 64, ids)
    assert (g["out"][:5] == 0).all()
    # out-of-range ids set the status bit and are treated as masked
    bad = ids.copy()
    bad[7, 0], bad[9, 2] = 99, -5
    wl = W.Workload("bad", P, Tr, E, k, 64, W.MOE_BF16, "uniform", "identity")
    x = W.draw_hidden(np.random.default_rng(1), wl.T, 64)
    w = np.random.default_rng(2).random((wl.T, k)).astype(np.float32)
    inp = W.Inputs(wl, x, None, bad, w, None)
    gg = run_gpu(wl, inp)
    from combine_top_histogram_gb300.binding import MOE_STATUS_BAD_EXPERT_ID
    assert gg["status"] == MOE_STATUS_BAD_EXPERT_ID
    oo = run_oracle(wl, inp)
    compare(wl, gg, oo, routed=False)
    # reading the status cleared it
    assert gg["layer"].status() == 0


@pytest.mark.parametrize("k", [1, 2, 3, 5, 8, 16, 32])
def test_edge_topk_values(gpu, k):
    rng = np.random.default_rng(k)
    P, Tr, E = 4, 29, 64
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)])
    _bf16_case(P, Tr, E, k, 128, ids, seed=k)


@pytest.mark.parametrize("P,Tr,E,k,H", [(1, 1, 1, 1, 8), (1, 513, 4, 2, 8), (64, 3, 128, 4, 24),
                                          (3, 1000, 3, 3, 1032), (16, 70, 1024, 8, 256)])
def test_edge_shapes(gpu, P, Tr, E, k, H):
    rng = np.random.default_rng(P * 7 + Tr)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)])
    _bf16_case(P, Tr, E, k, H, ids, seed=3)


def test_edge_duplicate_expert_in_one_token(gpu):
    P, Tr, E, k = 2, 19, 4, 3
    rng = np.random.default_rng(8)
    ids = rng.integers(0, E, (P * Tr, k))  # repeats allowed: (t, j) still orders them
    _bf16_case(P, Tr, E, k, 64, ids)


def test_edge_rank_reorder(gpu):
    """Swapping two ranks' token shards swaps their restored outputs."""
    P, Tr, E, k, H = 4, 50, 8, 2, 128
    rng = np.random.default_rng(9)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)])
    g1, _, _ = _bf16_case(P, Tr, E, k, H, ids, seed=10)
    wl = W.Workload("swap", P, Tr, E, k, H, W.MOE_BF16, "uniform", "identity", seed=10)
    rng2 = np.random.default_rng(10)
    x = W.draw_hidden(rng2, wl.T, H)
    w = rng2.random((wl.T, k)).astype(np.float32)
    perm = np.concatenate([np.arange(Tr, 2 * Tr), np.arange(0, Tr), np.arange(2 * Tr, P * Tr)])
    inp = W.Inputs(wl, x[perm].copy(), None, ids[perm].astype(np.int32), w[perm].copy(), None)
    g2 = run_gpu(wl, inp)
    assert np.array_equal(g2["out"], g1["out"][perm])


@pytest.mark.parametrize("cap", [1, 7, 64])
def test_fp8_capacity_parity(gpu, cap):
    wl = W.Workload("fp8cap", 4, 150, 16, 4, 384, W.MOE_FP8_E4M3, "uniform", "dequant",
                    cap=cap, seed=cap)
    inp = W.make_inputs(wl)
    inp.x[3, 128:256] = 0  # an all-zero 128-channel block
    _check(wl, inp)


@pytest.mark.parametrize("H,cap", [(256, 0), (512, 0), (1536, 1200)])
def test_fp8_dispatch_many_tokens_per_cta(gpu, H, cap):
    """More than 16 tokens per dispatch CTA (T = 40000 over at most 16 CTAs
    per SM): the FP8 dispatch stages each CTA's next row in shared memory
    while storing the current one; with H a multiple of 512 the receive rows
    are stored by bulk copies from shared memory (one with capacity drops).
    Every element against the oracle."""
    wl = W.UNIFORM_FP8.scaled(f"fp8_staged_{H}", Tr=5000, H=H, cap=cap)
    inp = W.make_inputs(wl)
    st = compare(wl, run_gpu(wl, inp), run_oracle(wl, inp), routed=False)
    if cap:
        assert st["kept"] < wl.Na


@pytest.mark.parametrize("name", ["uniform_fp8", "prefill_cap"])
def test_fp8_dispatch_with_x_only_16_byte_aligned(gpu, name):
    """x 16- but not 32-byte aligned: the FP8 dispatch takes its 16-byte-load
    kernel instead of the 32-byte one; both must match the oracle exactly."""
    wl = {"uniform_fp8": W.UNIFORM_FP8.scaled("u16", Tr=300, H=1024),
          "prefill_cap": W.PREFILL.scaled("p16", Tr=40, H=7168, cap=30)}[name]
    inp = W.make_inputs(wl)
    g = run_gpu(wl, inp, x_offset16=True)
    compare(wl, g, run_oracle(wl, inp), routed=inp.logits is not None)


def test_fp8_extreme_values(gpu):
    """Blocks with tiny, huge and mixed magnitudes (subnormal e4m3 codes,
    saturation at the amax element, negative zero after rounding)."""
    wl = W.Workload("fp8x", 2, 20, 4, 2, 512, W.MOE_FP8_E4M3, "uniform", "dequant", seed=7)
    inp = W.make_inputs(wl)
    rng = np.random.default_rng(0)
    vals = np.float32(rng.standard_normal((wl.T, wl.H))) * \
        np.float32(10.0) ** rng.integers(-30, 30, (wl.T, 1)).astype(np.float32)
    vals[:, :128] *= np.float32(1e-6) * (np.arange(128) % 2 == 0)  # wide dynamic range
    # blocks of subnormal values (bf16 keeps fp32's exponent range)
    vals[0, 128:256] = rng.standard_normal(128).astype(np.float32) * np.float32(1e-39)
    vals[1, 256:384] = np.float32(rng.integers(-3, 4, 128)) * np.float32(2.0 ** -133)
    vals[2, 384:512] = -0.0  # an all-zero block of negative zeros
    vals[3, 384:512] = np.where(np.arange(128) % 3 == 0, np.float32(-0.0), np.float32(1.5))
    inp.x[:] = W._bf16_bits_from_f32(vals.astype(np.float32))
    _check(wl, inp)


def test_layout_route_only_entry_point(gpu):
    import torch
    import oracle
    from combine_top_histogram_gb300 import binding as B
    wl = W.DECODE.scaled("r", Tr=21)
    inp = W.make_inputs(wl)
    h = B.moe_handle_create(B.make_config(wl.P, wl.Tr, wl.E, wl.k, wl.H))
    z = torch.from_numpy(inp.logits).cuda()
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    B.moe_route_topk(h, z, ids, w)
    oi, ow = oracle.route_topk(inp.logits, wl.k)
    assert np.array_equal(ids.cpu().numpy(), oi)
    from harness import f32_ulp_diff
    assert f32_ulp_diff(w.cpu().numpy(), ow).max() <= 1


ROUTE_CASES = [(256, 8), (64, 2), (8, 2), (1024, 32), (32, 1), (128, 5), (512, 16), (16, 8)]


@pytest.mark.parametrize("E,k", ROUTE_CASES, ids=[f"E{e}k{k}" for e, k in ROUTE_CASES])
def test_route_ties_gaps_and_chunkings(gpu, E, k):
    """Routing on logits with many exact ties (integers in [-3, 3] and rows of
    one repeated value: the lower expert wins), with large gaps (N(0, 40):
    weights far below 1, some under the float-float range) and N(0, 1), through
    the route-only kernel and the fused route+layout with one token per warp
    (small chunks) and several (large chunks): ids exact, weights within
    1 fp32 ulp of the double softmax."""
    import torch
    import oracle
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    from harness import f32_ulp_diff
    rng = np.random.default_rng(E * 100 + k)
    for Tr in (6, 2600):  # one token per routing warp / several per warp (T > 32 * SMs)
        P = 2
        T = P * Tr
        z = np.concatenate([
            rng.integers(-3, 4, (T // 3, E)).astype(np.float32),
            (rng.standard_normal((T // 3, E)) * 40).astype(np.float32),
            rng.standard_normal((T - 2 * (T // 3), E)).astype(np.float32)])
        z[0, :] = 0.5  # every logit equal
        oi, ow = oracle.route_topk(z, k)
        zt = torch.from_numpy(z).cuda()
        layer = MoeLayer(P, Tr, E, k, 128)
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        B.moe_route_topk(layer.handle, zt, ids, w)
        layer.route_layout(zt)
        torch.cuda.synchronize()
        for gi, gw in ((ids, w), (layer.ids, layer.w)):
            assert np.array_equal(gi.cpu().numpy(), oi), (Tr, E, k)
            assert f32_ulp_diff(gw.cpu().numpy(), ow).max() <= 1, (Tr, E, k)
        assert oi[0].tolist() == list(range(k))


def _threshold_boundary_logits(rng, n_tokens: int, extra: int) -> np.ndarray:
    """Logits (E = 256) whose top-8 threshold leaves exactly 32 + extra
    candidate keys: warp lane l holds experts l, l + 32, ..., l + 224, and
    eight lanes get four large logits each, the last of those lanes four
    equal ones (so the eighth-largest lane maximum is tied four ways); extra
    more large logits go to the first lane. Everything else is far below."""
    E = 256
    z = rng.standard_normal((n_tokens, E)).astype(np.float32)
    for t in range(n_tokens):
        lanes = rng.choice(32, 8, replace=False)
        regs = [rng.choice(8, 4 + (extra if q == 0 else 0), replace=False) for q in range(8)]
        tie = np.float32(10.0 + rng.random())
        for q, (lane, rs) in enumerate(zip(lanes, regs)):
            for i in rs:
                z[t, i * 32 + lane] = tie if q == 7 else np.float32(tie + 1.0 + rng.random())
    return z


def test_route_threshold_candidate_boundary(gpu):
    """The threshold top-k at its candidate limit: exactly 32 candidates (the
    compacted path, with a four-way tie at the threshold, the lower expert
    first) and 33 or more (the plain selection instead). Ids exact, weights
    within 1 fp32 ulp of the double softmax, through the route-only kernel
    and the fused route + layout."""
    import torch
    import oracle
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    from harness import f32_ulp_diff
    rng = np.random.default_rng(2026)
    P, Tr, E, k = 2, 300, 256, 8
    z = np.concatenate([_threshold_boundary_logits(rng, Tr, 0),
                        _threshold_boundary_logits(rng, Tr // 2, 1),
                        _threshold_boundary_logits(rng, Tr - Tr // 2, 4)])
    oi, ow = oracle.route_topk(z, k)
    zt = torch.from_numpy(z).cuda()
    layer = MoeLayer(P, Tr, E, k, 128)
    ids = torch.empty((P * Tr, k), dtype=torch.int32, device="cuda")
    w = torch.empty((P * Tr, k), dtype=torch.float32, device="cuda")
    B.moe_route_topk(layer.handle, zt, ids, w)
    layer.route_layout(zt)
    torch.cuda.synchronize()
    for gi, gw in ((ids, w), (layer.ids, layer.w)):
        assert np.array_equal(gi.cpu().numpy(), oi)
        assert f32_ulp_diff(gw.cpu().numpy(), ow).max() <= 1


def test_layout_tables_without_dispatch(gpu):
    """The per-source tables (cnt, kept counts, C, send and receive offsets)
    are left to the dispatch launch; moe_layout_tables builds them alone. With
    a capacity, 32 sources and 256 experts, every table equals the oracle's; a
    second call and a later dispatch (which then builds nothing) keep them."""
    import torch
    import oracle
    from combine_top_histogram_gb300 import MoeLayer
    from combine_top_histogram_gb300 import binding as B
    from harness import LAYOUT_KEYS
    wl = W.PREFILL.scaled("tables", Tr=50, H=128, cap=40)
    inp = W.make_inputs(wl)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    with pytest.raises(B.MoeError) as ei:
        layer.layout_tables()  # no layout yet
    assert ei.value.code == -5
    layer.route_layout(torch.from_numpy(inp.logits).cuda())
    layer.layout_tables()
    layer.layout_tables()
    torch.cuda.synchronize()
    ids = layer.ids.cpu().numpy()
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, ids, wl.cap)
    view = {k: v.cpu().numpy() for k, v in layer.layout_view().items()}
    checked = 0
    for gk, ok in LAYOUT_KEYS:
        if gk == "inv":
            continue
        assert np.array_equal(view[gk].reshape(-1), lay[ok].reshape(-1)), gk
        checked += 1
    assert checked >= 9
    assert view["totals"][:3].tolist() == lay["totals"].tolist()
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    layer.dispatch(x, layer.w)
    torch.cuda.synchronize()
    after = {k: v.cpu().numpy() for k, v in layer.layout_view().items()}
    assert np.array_equal(after["inv"].reshape(-1), lay["inv"].reshape(-1))
    for gk, _ in LAYOUT_KEYS:
        if gk != "inv":
            assert np.array_equal(after[gk], view[gk]), gk


def test_repeated_calls_on_one_handle(gpu):
    """The arrival counter resets itself: a second layer on the same handle
    (different routing) is as exact as the first."""
    from combine_top_histogram_gb300 import MoeLayer
    wl = W.UNIFORM_FP8.scaled("rep", Tr=600)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    for seed in (1, 2, 3):
        inp = W.make_inputs(wl, seed=seed)
        g = run_gpu(wl, inp, layer=layer)
        compare(wl, g, run_oracle(wl, inp), routed=False)


def test_errors_and_call_order(gpu):
    import torch
    from combine_top_histogram_gb300 import binding as B
    with pytest.raises(B.MoeError):
        B.moe_handle_create(B.make_config(3, 4, 8, 2, 64))  # E % P != 0
    with pytest.raises(B.MoeError):
        B.moe_handle_create(B.make_config(2, 4, 8, 2, 100, B.MOE_FP8_E4M3))  # H % 128
    h = B.moe_handle_create(B.make_config(2, 4, 8, 2, 64))
    y = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 2), dtype=torch.float32, device="cuda")
    out = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_combine(h, y, w, out)  # before any dispatch
    assert ei.value.code == -5
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.Handle(B.make_config(2, 4, 8, 2, 64), small)
    assert ei.value.code == -3


def test_host_copy_utilities(gpu):
    import torch
    from combine_top_histogram_gb300 import binding as B
    src = torch.arange(1 << 20, dtype=torch.int32).pin_memory()
    dev = torch.empty_like(src, device="cuda")
    back = torch.empty_like(src).pin_memory()
    B.moe_copy_h2d_async(dev, src)
    B.moe_copy_d2h_async(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    with pytest.raises(ValueError):
        B.moe_copy_h2d_async(dev[:10], src)


def test_fp8_quotients_at_e4m3_rounding_boundaries(gpu):
    """Blocks whose quotients x/s land exactly on, or one bf16 step around,
    e4m3 rounding boundaries (midpoints between neighbouring codes), with a
    power-of-two scale (exact quotients, ties to even) and inexact scales."""
    import oracle
    wl = W.Workload("fp8mid", 2, 8, 4, 2, 1024, W.MOE_FP8_E4M3, "uniform", "dequant", seed=11)
    inp = W.make_inputs(wl)
    reps = np.array([oracle.e4m3_value(c) for c in range(0x7F)], np.float64)
    mids = (reps[:-1] + reps[1:]) / 2
    rng = np.random.default_rng(12)
    vals = np.zeros((wl.T, wl.H), np.float32)
    for t in range(wl.T):
        for blk in range(wl.H // 128):
            amax = [56.0, 447.0, 3.0, 0.0371][(t + blk) % 4]  # s = amax / 448
            s = np.float32(np.float32(amax) / np.float32(448.0))
            m = rng.choice(mids, 127) * rng.choice([-1.0, 1.0], 127)
            x = (m * np.float64(s)).astype(np.float32)
            x *= np.float32(1.0) + np.float32(2.0 ** -8) * rng.integers(-1, 2, 127).astype(np.float32)
            row = np.concatenate([[amax], x]).astype(np.float32)
            vals[t, blk * 128:(blk + 1) * 128] = row
    inp.x[:] = W._bf16_bits_from_f32(vals)
    _check(wl, inp)
