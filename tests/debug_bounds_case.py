"""Runs in a child process with MOE_EP_DEBUG_BOUNDS=1, so the binding loads
the library built with device bounds checks (test_debug_bounds_gpu.py).

  clean    -- small layers in every dispatch mode: oracle parity, status 0
  corrupt  -- one expert offset in the workspace is overwritten (host side,
              between the layout and the dispatch) with a row past the
              receive buffer: the dispatch must skip that expert's rows, set
              MOE_STATUS_BOUNDS and leave every other row exact.
Exits 0 on success; refuses to run (exit 3) unless the loaded library reports
that it was built with the checks, so the corrupt case never reaches the
release kernels.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from combine_top_histogram_gb300 import binding as B  # noqa: E402
from combine_top_histogram_gb300 import workloads as W  # noqa: E402
from harness import compare, run_gpu, run_oracle, to_np_bits  # noqa: E402


def clean():
    cases = [(W.SKEWED.scaled("dbg_skewed", Tr=200, H=256), dict()),
             (W.PREFILL.scaled("dbg_prefill", Tr=30, H=256, cap=32), dict()),
             (W.SKEWED.scaled("dbg_two_stage", Tr=200, H=256), dict(two_stage=True)),
             (W.PREFILL.scaled("dbg_allgather", Tr=30, H=256, cap=32), dict(allgather=True)),
             (W.DECODE.scaled("dbg_fused", Tr=37, H=512), dict(fused=True)),
             (W.UNIFORM_FP8.scaled("dbg_pipelined", Tr=300, H=256), dict(pipelined=3))]
    for wl, flags in cases:
        inp = W.make_inputs(wl)
        g = run_gpu(wl, inp, **flags)
        o = run_oracle(wl, inp)
        compare(wl, g, o, routed=inp.logits is not None)
        assert g["status"] == 0, (wl.name, g["status"])
        print("clean", wl.name, "ok", flush=True)


def corrupt():
    import torch
    from combine_top_histogram_gb300 import MoeLayer
    wl = W.Workload("dbg_corrupt", 4, 64, 16, 2, 256, W.MOE_BF16, "uniform", "identity", seed=9)
    inp = W.make_inputs(wl)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap, "cuda:0")
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(inp.ids).cuda()
    w = torch.from_numpy(inp.w).cuda()
    bad_e = 5
    layer.layout(ids)
    # the layout tables first: the layout is then scanned, and the dispatch
    # reads the expert offsets from the workspace (a small layout would
    # otherwise be dispatched directly from the per-expert totals)
    layer.layout_tables()
    view = layer.layout_view()
    view["expert_offset"][bad_e] = layer.rows + 5  # past the receive buffer
    layer.dispatch(x, w)
    layer.expert()
    layer.combine(w)
    torch.cuda.synchronize()
    st = layer.status()
    assert st & B.MOE_STATUS_BOUNDS, hex(st)
    lay = oracle.layout(wl.P, wl.Tr, wl.E, wl.k, inp.ids, 0)
    inv = to_np_bits(layer.layout_view()["inv"])
    flat = inp.ids.reshape(-1)
    assert (inv[flat == bad_e] == -1).all()
    ok = flat != bad_e
    assert np.array_equal(inv[ok], lay["inv"][ok])
    # a clean layer afterwards on the same handle (direct dispatch) is exact again
    layer.layout(ids)
    layer.dispatch(x, w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(to_np_bits(layer.layout_view()["inv"]), lay["inv"])
    print("corrupt ok", flush=True)


if __name__ == "__main__":
    if not (B.library_path().endswith("libmoe_ep_debug.so") and B.moe_debug_bounds()):
        print("not the bounds-checked library", flush=True)
        sys.exit(3)
    {"clean": clean, "corrupt": corrupt}[sys.argv[1]]()
