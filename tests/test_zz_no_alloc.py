"""The no-allocation layout entry point against the workspace path.

moe_dispatch_layout_noalloc exists for callers that cannot allocate device
memory (graph capture in progress, plugin interfaces without a workspace,
externally owned allocators). Its scratch is a static device array shared by
every call, so this test makes two calls in a row with different routings and
capacities and checks each, through the C ABI, against what the handle-based
path (moe_dispatch_layout + moe_dispatch) computes on the same ids: every
count, offset and the inverse permutation, bit for bit. This file is named to
be collected last.
"""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NAMES = ["expert_count", "expert_count_raw", "expert_offset", "src_expert_count",
         "src_expert_kept", "count_matrix", "send_offset", "recv_offset", "rank_base", "inv",
         "totals"]


def _workspace_path(wl, ids_np, w_np):
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    x = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    layer.layout(ids)
    layer.dispatch(x, w)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().copy() for k, v in layer.layout_view().items()}


def _noalloc_path(wl, ids_np):
    import torch
    from combine_top_histogram_gb300 import binding as B
    P, E, Na = wl.P, wl.E, wl.Na
    shapes = dict(expert_count=(E,), expert_count_raw=(E,), expert_offset=(E + 1,),
                  src_expert_count=(P, E), src_expert_kept=(P, E), count_matrix=(P, P),
                  send_offset=(P, P), recv_offset=(P, E), rank_base=(P + 1,), inv=(Na,),
                  totals=(4,))
    # poison the outputs so an unwritten element cannot pass
    out = {k: torch.full(s, -777, dtype=torch.int32, device="cuda") for k, s in shapes.items()}
    cfg = B.make_config(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    B.moe_dispatch_layout_noalloc(cfg, torch.from_numpy(ids_np).cuda(), out)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_noalloc_layout_matches_workspace_path_twice(gpu):
    calls = [
        (W.UNIFORM_FP8.scaled("noalloc_a", Tr=1100, H=128), 1, 0.0),
        (W.PREFILL.scaled("noalloc_b", Tr=100, H=128, cap=90), 2, 0.1),
    ]
    for wl, seed, mask in calls:
        rng = np.random.default_rng(seed)
        ids = np.stack([rng.permutation(wl.E)[:wl.k] for _ in range(wl.T)]).astype(np.int32)
        ids = W.mask_random_slots(ids, mask, seed)
        w = rng.random((wl.T, wl.k)).astype(np.float32)
        want = _workspace_path(wl, ids, w)
        got = _noalloc_path(wl, ids)
        for name in NAMES:
            a, b = got[name].reshape(-1), want[name].reshape(-1)
            if name == "totals":
                a, b = a[:3], b[:3]
            assert np.array_equal(a, b), (wl.name, name)


def test_noalloc_rejects_sizes_beyond_its_scratch(gpu):
    import torch
    from combine_top_histogram_gb300 import binding as B
    wl = W.PREFILL.scaled("too_big", Tr=8192, H=128)  # 2,097,152 assignments > 8 MiB of codes
    cfg = B.make_config(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    out = {n: torch.zeros(1, dtype=torch.int32, device="cuda") for n in NAMES}
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_dispatch_layout_noalloc(cfg, ids, out)
    assert ei.value.code == -2
