"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/moe_ep.h declares; host-only entry points validate their arguments
without touching a GPU."""
import ctypes
import os
import re

from combine_top_histogram_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "moe_ep.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(B.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(cuda_lib):
    for name in declared_functions():
        assert hasattr(cuda_lib, name), name
    out = os.popen(f"nm -D --defined-only {B.library_path()}").read()
    exported = set(re.findall(r"\bT (moe_[a-z_0-9]+)", out))
    assert set(declared_functions()) <= exported


def test_debug_build_exports_the_same_symbols_and_reports_its_checks(cuda_lib):
    import importlib
    build = importlib.import_module("combine_top_histogram_gb300.build")
    build.build(variants=("debug",))
    out = os.popen(f"nm -D --defined-only {build.DEBUG_LIB_PATH}").read()
    exported = set(re.findall(r"\bT (moe_[a-z_0-9]+)", out))
    assert set(declared_functions()) <= exported
    dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
    assert dbg.moe_debug_bounds() == 1
    assert cuda_lib.moe_debug_bounds() == 0


def test_host_only_sizing_and_validation(cuda_lib):
    cfg = B.make_config(8, 128, 256, 8, 7168)
    assert B.moe_recv_rows_max(cfg) == 8 * 128 * 8
    capped = B.make_config(32, 4096, 256, 8, 7168, B.MOE_FP8_E4M3, 5120)
    assert B.moe_recv_rows_max(capped) == min(32 * 4096 * 8, 256 * 5120)
    assert B.moe_recv_rows_max(B.make_config(4, 2, 8, 2, 128, cap=1)) == 8
    nbytes = B.moe_workspace_bytes(cfg)
    assert nbytes >= 2 * 8 * 128 * 8 * 4  # assignment codes and inv
    for bad in [B.make_config(3, 4, 8, 2, 64), B.make_config(2, 4, 8, 9, 64),
                B.make_config(2, 4, 8, 2, 12), B.make_config(2, 4, 2048, 2, 64),
                B.make_config(2, 4, 8, 2, 64, B.MOE_FP8_E4M3), B.make_config(0, 4, 8, 2, 64),
                B.make_config(2, 4, 8, 2, 64, cap=-1), B.make_config(2, 4, 64, 33, 64),
                B.make_config(1024, 1, 1024, 1, 64), B.make_config(256, 2, 512, 2, 64)]:
        assert B.moe_workspace_bytes(bad) == 0
        assert B.moe_recv_rows_max(bad) == 0
        h = ctypes.c_void_p()
        rc = cuda_lib.moe_handle_create(ctypes.byref(bad), ctypes.c_void_p(256), 1 << 20,
                                        ctypes.byref(h))
        assert rc in (-1, -2) and not h.value
    assert B.moe_error_string(-3) == "workspace too small or misaligned"
    assert cuda_lib.moe_handle_destroy(None) == 0


def test_fixed_slot_rows_rule():
    from combine_top_histogram_gb300 import binding as B
    assert B.moe_fixed_slot_rows(B.make_config(8, 128, 256, 8, 7168)) == 256 * 8 * 128
    assert B.moe_fixed_slot_rows(B.make_config(4, 2, 8, 2, 128)) == 8 * 4 * 2
    assert B.moe_fixed_slot_rows(B.make_config(8, 128, 256, 8, 7168, cap=64)) == 0  # capacity
    assert B.moe_fixed_slot_rows(B.make_config(32, 1 << 20, 256, 8, 128)) == 0  # > int32 rows
    assert B.moe_fixed_slot_rows(B.make_config(3, 4, 8, 2, 64)) == 0  # invalid config


def test_null_handles_are_rejected(cuda_lib):
    assert cuda_lib.moe_dispatch_layout(None, None, None) == -1
    assert cuda_lib.moe_combine(None, None, None, None, None) == -1
    assert cuda_lib.moe_route_topk(None, None, None, None, None) == -1
    assert cuda_lib.moe_layout_tables(None, None) == -1


def test_build_targets_sm103a_without_fast_math():
    import importlib
    bld = importlib.import_module("combine_top_histogram_gb300.build")
    assert bld.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "use_fast_math" not in open(bld.__file__).read()
