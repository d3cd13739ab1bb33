"""Runs one workload through the CUDA library and through the CPU oracle on the
same seeded inputs, and compares the results element by element."""
from __future__ import annotations

import numpy as np

import oracle
from combine_top_histogram_gb300 import workloads as W

LAYOUT_KEYS = [  # (library view name, oracle name)
    ("expert_count", "n_kept"), ("expert_count_raw", "n_raw"),
    ("expert_offset", "expert_offset"), ("src_expert_count", "cnt"),
    ("src_expert_kept", "kept_cnt"), ("count_matrix", "C"), ("send_offset", "send_offset"),
    ("recv_offset", "recv_offset"), ("rank_base", "rank_base"), ("inv", "inv")]
META_KEYS = ["local_expert", "src_rank", "src_token", "slot", "weight"]


def to_np_bits(t):
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_gpu(wl: W.Workload, inp: W.Inputs, ids=None, layer=None, stream=None,
            copy_rows: bool = True, two_stage: bool = False, fused: bool = False,
            pipelined: int = 0, allgather: bool = False, x_offset16: bool = False):
    """The path on the GPU through the C ABI; returns host copies of everything
    (copy_rows=False leaves the row buffers on the device, in res["layer"]).
    x_offset16: x starts 16 bytes past a 256-byte boundary (16-byte aligned,
    not 32-byte aligned), which selects the dispatch's 16-byte-load kernels."""
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    dev = torch.device("cuda:0")
    if layer is None:
        layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap, "cuda:0")
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    if x_offset16:
        buf = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device=dev)
        buf[8:].copy_(x.reshape(-1))
        x = buf[8:].view(x.shape)
        assert x.data_ptr() % 32 == 16
    c = torch.from_numpy(inp.expert_scale).to(dev) if inp.expert_scale is not None else None
    if pipelined:
        if ids is None and inp.logits is not None:
            layer.forward_pipelined(x, logits=torch.from_numpy(inp.logits).to(dev), expert_scale=c,
                                    chunks=pipelined)
            w_used = layer.w
        else:
            ids_np = inp.ids if ids is None else ids
            w_used = torch.from_numpy(inp.w).to(dev)
            layer.forward_pipelined(x, ids=torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).to(dev),
                                    w=w_used, expert_scale=c, chunks=pipelined)
    elif ids is None and inp.logits is not None:
        logits = torch.from_numpy(inp.logits).to(dev)
        layer.forward(x, logits=logits, expert_scale=c, stream=stream, two_stage=two_stage,
                      fused=fused, allgather=allgather)
        w_used = layer.w
    else:
        ids_np = inp.ids if ids is None else ids
        ids_t = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).to(dev)
        w_used = torch.from_numpy(inp.w).to(dev)
        layer.forward(x, ids=ids_t, w=w_used, expert_scale=c, stream=stream, two_stage=two_stage,
                      fused=fused, allgather=allgather)
    torch.cuda.synchronize()
    view = layer.layout_view()
    res = {k: to_np_bits(v) for k, v in view.items()}
    res["ids"] = to_np_bits(layer.ids) if inp.logits is not None and ids is None else None
    res["w"] = to_np_bits(w_used)
    if copy_rows:
        res["recv_x"] = to_np_bits(layer.recv_x)
        res["recv_scale"] = to_np_bits(layer.recv_scale) if layer.recv_scale is not None else None
        res["meta"] = {k: to_np_bits(v) for k, v in layer.meta.items()}
        res["y"] = to_np_bits(layer.y)
        res["out"] = to_np_bits(layer.out)
    res["status"] = layer.status()
    res["layer"] = layer
    return res


def run_oracle(wl: W.Workload, inp: W.Inputs, ids=None, w=None, threads: int = 1):
    """The same layer on the CPU oracle. ids/w override the inputs' routing.
    threads > 1 runs the oracle's token-independent steps on token ranges."""
    if ids is None and inp.logits is not None:
        ids, w = oracle.route_topk(inp.logits, wl.k, threads=threads)
    elif ids is None:
        ids, w = inp.ids, inp.w
    elif w is None:
        w = inp.w
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, ids, wl.cap)
    rows = wl.rows_max
    fp8 = wl.dispatch_dtype == W.MOE_FP8_E4M3
    if fp8:
        recv, sc, meta = oracle.dispatch_fp8(wl.P, wl.Tr, wl.E, wl.k, inp.x, w, ids, lay["inv"],
                                             rows, threads=threads)
        y = oracle.expert_dequant_fp8(recv, sc, threads=threads)
    else:
        recv, meta = oracle.dispatch_bf16(wl.P, wl.Tr, wl.E, wl.k, inp.x, w, ids, lay["inv"],
                                          rows, threads=threads)
        sc = None
        c = inp.expert_scale if inp.expert_scale is not None else np.ones(wl.E, np.float32)
        y = oracle.expert_scale_bf16(wl.E, lay["expert_offset"], c, recv)
    out = oracle.combine(lay["inv"], w, y, wl.T, wl.k, threads=threads)
    return dict(ids=ids, w=w, layout=lay, recv_x=recv, recv_scale=sc, meta=meta, y=y, out=out)


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (monotone integer mapping)."""
    def key(b):
        v = b.astype(np.int32)
        return np.where(v & 0x8000, 0x8000 - (v & 0x7FFF), 0x8000 + v)
    return np.abs(key(a_bits) - key(b_bits))


def f32_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def key(x):
        v = np.ascontiguousarray(x, np.float32).view(np.int32).astype(np.int64)
        return np.where(v < 0, -(v & 0x7FFFFFFF), v)
    return np.abs(key(a) - key(b))


def compare(wl: W.Workload, g: dict, o: dict, routed: bool):
    """Asserts the parity bar: bit-exact layout, permutation, metadata, payload
    and FP8 codes/scales; route weights within 1 fp32 ulp; combine within
    1 bf16 ulp. Returns a few statistics."""
    stats = {}
    if routed:
        assert np.array_equal(g["ids"], o["ids"]), "route ids differ"
        d = f32_ulp_diff(g["w"], o["w"])
        assert d.max() <= 1, f"route weights differ by {d.max()} ulp"
        stats["route_w_exact"] = float((d == 0).mean())
    lay = o["layout"]
    for gk, ok in LAYOUT_KEYS:
        assert np.array_equal(g[gk].reshape(-1), lay[ok].reshape(-1)), f"layout {gk} differs"
    assert g["totals"][:3].tolist() == lay["totals"].tolist(), "totals differ"
    n = int(lay["totals"][0])
    assert np.array_equal(g["recv_x"][:n], o["recv_x"][:n]), "dispatch payload differs"
    if o["recv_scale"] is not None:
        assert np.array_equal(g["recv_scale"][:n].view(np.uint32),
                              o["recv_scale"][:n].view(np.uint32)), "fp8 scales differ"
    for k in META_KEYS:
        a, b = g["meta"][k][:n], o["meta"][k][:n]
        if k == "weight":
            # routed weights may differ by 1 fp32 ulp (double exp on both sides)
            tol = 1 if routed else 0
            assert f32_ulp_diff(a, b).max() <= tol, "meta weight differs"
        else:
            assert np.array_equal(a, b), f"meta {k} differs"
    assert np.array_equal(g["y"][:n], o["y"][:n]), "expert stand-in differs"
    d = bf16_ulp_diff(g["out"], o["out"])
    assert d.max() <= 1, f"combine differs by {d.max()} bf16 ulp"
    stats["combine_exact"] = float((d == 0).mean())
    stats["kept"] = n
    return stats
