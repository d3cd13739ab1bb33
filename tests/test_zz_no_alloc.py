"""The no-allocation layout entry point, through the C ABI.

moe_dispatch_layout_noalloc serves callers that may not call cudaMalloc and
have no workspace to hand over (plugin interfaces that pass only inputs and
outputs, processes whose device memory belongs to another allocator, code
that must not let an allocation synchronise the device). Its scratch is a
static device array shared by every call, so the test makes two calls in a
row with different routings and capacities and checks each, bit for bit,
against the oracle's layout and against what the handle-based path
(moe_dispatch_layout + moe_dispatch) computes on the same ids: every count,
offset and the inverse permutation. It also checks that a call allocates no
device memory, and that sizes beyond the scratch or the layout kernels'
shared memory are refused before anything is enqueued. This file is named to
be collected last.
"""
import numpy as np
import pytest

import oracle
from combine_top_histogram_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NAMES = ["expert_count", "expert_count_raw", "expert_offset", "src_expert_count",
         "src_expert_kept", "count_matrix", "send_offset", "recv_offset", "rank_base", "inv",
         "totals"]
ORACLE_NAME = {"expert_count": "n_kept", "expert_count_raw": "n_raw",
               "expert_offset": "expert_offset", "src_expert_count": "cnt",
               "src_expert_kept": "kept_cnt", "count_matrix": "C", "send_offset": "send_offset",
               "recv_offset": "recv_offset", "rank_base": "rank_base", "inv": "inv",
               "totals": "totals"}


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


def _outputs(wl):
    import torch
    P, E, Na = wl.P, wl.E, wl.Na
    shapes = dict(expert_count=(E,), expert_count_raw=(E,), expert_offset=(E + 1,),
                  src_expert_count=(P, E), src_expert_kept=(P, E), count_matrix=(P, P),
                  send_offset=(P, P), recv_offset=(P, E), rank_base=(P + 1,), inv=(Na,),
                  totals=(4,))
    # poisoned, so that an unwritten element cannot pass
    return {k: torch.full(s, -777, dtype=torch.int32, device="cuda") for k, s in shapes.items()}


def _noalloc_path(wl, ids_np, out=None):
    import torch
    from combine_top_histogram_gb300 import binding as B
    out = _outputs(wl) if out is None else out
    cfg = B.make_config(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    B.moe_dispatch_layout_noalloc(cfg, torch.from_numpy(ids_np).cuda(), out)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _ids(wl, seed, mask):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(wl.E)[:wl.k] for _ in range(wl.T)]).astype(np.int32)
    ids = W.mask_random_slots(ids, mask, seed)
    w = rng.random((wl.T, wl.k)).astype(np.float32)
    return ids, w


def test_noalloc_layout_matches_oracle_and_workspace_path_twice(gpu):
    calls = [
        (W.UNIFORM_FP8.scaled("noalloc_a", Tr=1100, H=128), 1, 0.0),
        (W.PREFILL.scaled("noalloc_b", Tr=100, H=128, cap=90), 2, 0.1),
    ]
    for wl, seed, mask in calls:
        ids, w = _ids(wl, seed, mask)
        got = _noalloc_path(wl, ids)
        want_o = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, ids, wl.cap)
        want_w = _workspace_path(wl, ids, w)
        for name in NAMES:
            a = got[name].reshape(-1)
            o = want_o[ORACLE_NAME[name]].reshape(-1)
            b = want_w[name].reshape(-1)
            if name == "totals":
                a, b = a[:3], b[:3]
            assert np.array_equal(a, o), (wl.name, name, "oracle")
            assert np.array_equal(a, b), (wl.name, name, "workspace path")
        if wl.cap:
            assert got["totals"][1] > 0  # the capacity dropped rows


def test_noalloc_call_allocates_no_device_memory(gpu):
    import torch
    wl = W.DECODE.scaled("noalloc_mem", Tr=300, H=128)
    ids1, _ = _ids(wl, 3, 0.05)
    ids2, _ = _ids(wl, 4, 0.0)
    out = _outputs(wl)
    ids2_d = torch.from_numpy(ids2).cuda()
    _noalloc_path(wl, ids1, out)  # set-up and kernel loading happen here
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    from combine_top_histogram_gb300 import binding as B
    cfg = B.make_config(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap)
    B.moe_dispatch_layout_noalloc(cfg, ids2_d, out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, ids2, wl.cap)
    assert np.array_equal(out["inv"].cpu().numpy(), lay["inv"])


def test_noalloc_rejects_sizes_beyond_its_limits(gpu):
    import torch
    from combine_top_histogram_gb300 import binding as B
    out = {n: torch.zeros(1, dtype=torch.int32, device="cuda") for n in NAMES}
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 2,097,152 assignments: 8 MiB of codes alone, beyond the scratch
    wl = W.PREFILL.scaled("too_big", Tr=8192, H=128)
    # 512 ranks x 512 experts, one token each: the scratch fits (about 2 MB),
    # but the scan's per-(source, expert) table (about 2 MB) exceeds shared memory
    wide = W.Workload("too_wide", 512, 1, 512, 1, 128, W.MOE_BF16, "uniform", "identity")
    for w_ in (wl, wide):
        cfg = B.make_config(w_.P, w_.Tr, w_.E, w_.k, w_.H, w_.dispatch_dtype, w_.cap)
        with pytest.raises(B.MoeError) as ei:
            B.moe_dispatch_layout_noalloc(cfg, ids, out)
        assert ei.value.code == -2, w_.name
