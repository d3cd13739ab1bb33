"""Thin ctypes binding of libmoe_ep.so (include/moe_ep.h).

Argument marshalling only: every function passes torch tensors' device
pointers and the current CUDA stream to the C entry point of the same name and
raises MoeError on a negative return code. No step of the path runs here.
If the library has not been built, loading it raises immediately: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import build as _build

MOE_BF16 = 0
MOE_FP8_E4M3 = 1
MOE_STATUS_BAD_EXPERT_ID = 0x1
MOE_STATUS_TIMEOUT = 0x2
MOE_STATUS_SLOT_OVERFLOW = 0x4
MOE_STATUS_BOUNDS = 0x8
MOE_MAX_EXPERTS = 1024
MOE_MAX_TOPK = 32
MOE_MAX_RANKS = 1024

_c_void_p = ctypes.c_void_p

#: Every symbol include/moe_ep.h declares.
EXPORTED_SYMBOLS = (
    "moe_workspace_bytes", "moe_recv_rows_max", "moe_handle_create", "moe_handle_destroy",
    "moe_route_topk", "moe_dispatch_layout", "moe_route_dispatch_layout", "moe_get_layout",
    "moe_dispatch", "moe_expert_standin", "moe_combine", "moe_read_status", "moe_error_string",
    "moe_dispatch_layout_noalloc", "moe_copy_h2d_async", "moe_copy_d2h_async",
    "moe_dispatch_two_stage", "moe_layout_dispatch_fused", "moe_set_wait_limit",
    "moe_dispatch_tokens", "moe_expert_standin_tokens", "moe_combine_tokens",
    "moe_dispatch_allgather", "moe_layout_tables", "moe_dispatch_fixed_slots",
    "moe_fixed_slot_rows", "moe_debug_bounds",
)


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


class moe_config_t(ctypes.Structure):
    _fields_ = [("num_ranks", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("dispatch_dtype", ctypes.c_int32),
                ("combine_dtype", ctypes.c_int32), ("expert_capacity", ctypes.c_int32)]


class moe_layout_view_t(ctypes.Structure):
    _fields_ = [(n, _c_void_p) for n in (
        "expert_count", "expert_count_raw", "expert_offset", "src_expert_count",
        "src_expert_kept", "count_matrix", "send_offset", "recv_offset", "rank_base", "inv",
        "totals")]


class moe_recv_meta_t(ctypes.Structure):
    _fields_ = [(n, _c_void_p) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    """The release library; with MOE_EP_DEBUG_BOUNDS=1 in the environment the
    build with device bounds checks (MOE_STATUS_BOUNDS); with MOE_EP_LIBRARY
    set, that file (another build of the same sources)."""
    if os.environ.get("MOE_EP_LIBRARY"):
        return os.environ["MOE_EP_LIBRARY"]
    if os.environ.get("MOE_EP_DEBUG_BOUNDS", "") == "1":
        return _build.DEBUG_LIB_PATH
    return _build.LIB_PATH


def load_library():
    """Loads the built library; raises if it is missing (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"libmoe_ep.so is not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        i32, sz, vp = ctypes.c_int, ctypes.c_size_t, _c_void_p
        cfgp = ctypes.POINTER(moe_config_t)
        lib.moe_workspace_bytes.restype = sz
        lib.moe_workspace_bytes.argtypes = [cfgp]
        lib.moe_recv_rows_max.restype = ctypes.c_int64
        lib.moe_recv_rows_max.argtypes = [cfgp]
        lib.moe_handle_create.restype = i32
        lib.moe_handle_create.argtypes = [cfgp, vp, sz, ctypes.POINTER(vp)]
        lib.moe_handle_destroy.restype = i32
        lib.moe_handle_destroy.argtypes = [vp]
        lib.moe_route_topk.restype = i32
        lib.moe_route_topk.argtypes = [vp, vp, vp, vp, vp]
        lib.moe_dispatch_layout.restype = i32
        lib.moe_dispatch_layout.argtypes = [vp, vp, vp]
        lib.moe_route_dispatch_layout.restype = i32
        lib.moe_route_dispatch_layout.argtypes = [vp, vp, vp, vp, vp]
        lib.moe_dispatch_fixed_slots.restype = i32
        lib.moe_dispatch_fixed_slots.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_fixed_slot_rows.restype = ctypes.c_int64
        lib.moe_fixed_slot_rows.argtypes = [cfgp]
        lib.moe_layout_tables.restype = i32
        lib.moe_layout_tables.argtypes = [vp, vp]
        lib.moe_get_layout.restype = i32
        lib.moe_get_layout.argtypes = [vp, ctypes.POINTER(moe_layout_view_t)]
        lib.moe_dispatch.restype = i32
        lib.moe_dispatch.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_dispatch_two_stage.restype = i32
        lib.moe_dispatch_two_stage.argtypes = [vp, vp, vp, vp, vp, vp, vp,
                                               ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_layout_dispatch_fused.restype = i32
        lib.moe_layout_dispatch_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp,
                                                  ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_set_wait_limit.restype = i32
        lib.moe_set_wait_limit.argtypes = [vp, ctypes.c_int64]
        i64 = ctypes.c_int64
        lib.moe_dispatch_tokens.restype = i32
        lib.moe_dispatch_tokens.argtypes = [vp, i64, i64, vp, vp, vp, vp,
                                            ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_expert_standin_tokens.restype = i32
        lib.moe_expert_standin_tokens.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp]
        lib.moe_combine_tokens.restype = i32
        lib.moe_combine_tokens.argtypes = [vp, i64, i64, vp, vp, vp, vp]
        lib.moe_dispatch_allgather.restype = i32
        lib.moe_dispatch_allgather.argtypes = [vp, vp, vp, vp, vp, vp, vp,
                                               ctypes.POINTER(moe_recv_meta_t), vp]
        lib.moe_expert_standin.restype = i32
        lib.moe_expert_standin.argtypes = [vp, vp, vp, vp, vp, vp]
        lib.moe_combine.restype = i32
        lib.moe_combine.argtypes = [vp, vp, vp, vp, vp]
        lib.moe_read_status.restype = i32
        lib.moe_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.moe_dispatch_layout_noalloc.restype = i32
        lib.moe_dispatch_layout_noalloc.argtypes = [cfgp, vp, ctypes.POINTER(moe_layout_view_t), vp]
        lib.moe_copy_h2d_async.restype = i32
        lib.moe_copy_h2d_async.argtypes = [vp, vp, sz, vp]
        lib.moe_copy_d2h_async.restype = i32
        lib.moe_copy_d2h_async.argtypes = [vp, vp, sz, vp]
        lib.moe_error_string.restype = ctypes.c_char_p
        lib.moe_error_string.argtypes = [i32]
        lib.moe_debug_bounds.restype = i32
        lib.moe_debug_bounds.argtypes = []
        _lib = lib
        return lib


def _check(fn: str, rc: int) -> None:
    if rc < 0:
        raise MoeError(fn, rc, load_library().moe_error_string(rc).decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(P: int, Tr: int, E: int, k: int, H: int, dispatch_dtype: int = MOE_BF16,
                cap: int = 0) -> moe_config_t:
    return moe_config_t(P, Tr, E, k, H, dispatch_dtype, MOE_BF16, cap)


def moe_workspace_bytes(cfg: moe_config_t) -> int:
    return int(load_library().moe_workspace_bytes(ctypes.byref(cfg)))


def moe_recv_rows_max(cfg: moe_config_t) -> int:
    return int(load_library().moe_recv_rows_max(ctypes.byref(cfg)))


class Handle:
    """Owns the C handle and keeps its workspace tensor alive."""

    def __init__(self, cfg: moe_config_t, workspace):
        self.cfg = cfg
        self.workspace = workspace
        h = _c_void_p()
        _check("moe_handle_create", load_library().moe_handle_create(
            ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
            ctypes.byref(h)))
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self):
        if self._h:
            load_library().moe_handle_destroy(self._h)
            self._h = _c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_handle_create(cfg: moe_config_t, workspace=None, device=None) -> Handle:
    """Creates a handle; allocates the workspace with torch when none is given."""
    import torch
    if workspace is None:
        nbytes = moe_workspace_bytes(cfg)
        if nbytes == 0:
            _check("moe_workspace_bytes", -1)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    return Handle(cfg, workspace)


def moe_route_topk(h: Handle, logits, ids, w, stream=None) -> None:
    _check("moe_route_topk", load_library().moe_route_topk(
        h.ptr, _ptr(logits), _ptr(ids), _ptr(w), _stream(stream)))


def moe_dispatch_layout(h: Handle, ids, stream=None) -> None:
    _check("moe_dispatch_layout", load_library().moe_dispatch_layout(
        h.ptr, _ptr(ids), _stream(stream)))


def moe_route_dispatch_layout(h: Handle, logits, ids, w, stream=None) -> None:
    _check("moe_route_dispatch_layout", load_library().moe_route_dispatch_layout(
        h.ptr, _ptr(logits), _ptr(ids), _ptr(w), _stream(stream)))


def moe_fixed_slot_rows(cfg) -> int:
    return int(load_library().moe_fixed_slot_rows(ctypes.byref(cfg)))


def moe_dispatch_fixed_slots(h: Handle, x, w, slot_x, slot_scale, meta: dict, stream=None) -> None:
    """Dispatch into fixed per-(source, expert) slot regions (see the header)."""
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_dispatch_fixed_slots", load_library().moe_dispatch_fixed_slots(
        h.ptr, _ptr(x), _ptr(w), _ptr(slot_x), _ptr(slot_scale), ctypes.byref(m),
        _stream(stream)))


def moe_layout_tables(h: Handle, stream=None) -> None:
    """Completes the per-source tables of the last layout without dispatching."""
    _check("moe_layout_tables", load_library().moe_layout_tables(h.ptr, _stream(stream)))


def moe_get_layout(h: Handle) -> dict:
    """Views (int32 tensors on the workspace) of every layout array."""
    import torch
    v = moe_layout_view_t()
    _check("moe_get_layout", load_library().moe_get_layout(h.ptr, ctypes.byref(v)))
    cfg = h.cfg
    P, E = cfg.num_ranks, cfg.num_experts
    Na = P * cfg.tokens_per_rank * cfg.top_k
    sizes = dict(expert_count=(E,), expert_count_raw=(E,), expert_offset=(E + 1,),
                 src_expert_count=(P, E), src_expert_kept=(P, E), count_matrix=(P, P),
                 send_offset=(P, P), recv_offset=(P, E), rank_base=(P + 1,), inv=(Na,),
                 totals=(4,))
    ws = h.workspace
    base = ws.data_ptr()
    out = {}
    for name, shape in sizes.items():
        off = getattr(v, name) - base
        n = 1
        for s in shape:
            n *= s
        out[name] = ws[off: off + 4 * n].view(torch.int32).view(*shape)
    return out


def moe_dispatch(h: Handle, x, w, recv_x, recv_scale, meta: dict, stream=None) -> None:
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_dispatch", load_library().moe_dispatch(
        h.ptr, _ptr(x), _ptr(w), _ptr(recv_x), _ptr(recv_scale), ctypes.byref(m),
        _stream(stream)))


def moe_dispatch_two_stage(h: Handle, x, w, send_x, send_scale, recv_x, recv_scale, meta: dict,
                           stream=None) -> None:
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_dispatch_two_stage", load_library().moe_dispatch_two_stage(
        h.ptr, _ptr(x), _ptr(w), _ptr(send_x), _ptr(send_scale), _ptr(recv_x), _ptr(recv_scale),
        ctypes.byref(m), _stream(stream)))


def moe_layout_dispatch_fused(h: Handle, logits, ids, w, x, recv_x, recv_scale, meta: dict,
                              stream=None) -> None:
    """Route (logits given) or take ids/w, lay out and dispatch in one launch."""
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_layout_dispatch_fused", load_library().moe_layout_dispatch_fused(
        h.ptr, _ptr(logits), _ptr(ids), _ptr(w), _ptr(x), _ptr(recv_x), _ptr(recv_scale),
        ctypes.byref(m), _stream(stream)))


def moe_set_wait_limit(h: Handle, polls: int) -> None:
    _check("moe_set_wait_limit", load_library().moe_set_wait_limit(h.ptr, int(polls)))


def moe_dispatch_tokens(h: Handle, begin: int, end: int, x, w, recv_x, recv_scale, meta: dict,
                        stream=None) -> None:
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_dispatch_tokens", load_library().moe_dispatch_tokens(
        h.ptr, int(begin), int(end), _ptr(x), _ptr(w), _ptr(recv_x), _ptr(recv_scale),
        ctypes.byref(m), _stream(stream)))


def moe_expert_standin_tokens(h: Handle, begin: int, end: int, recv_x, recv_scale, expert_scale,
                              y, stream=None) -> None:
    _check("moe_expert_standin_tokens", load_library().moe_expert_standin_tokens(
        h.ptr, int(begin), int(end), _ptr(recv_x), _ptr(recv_scale), _ptr(expert_scale),
        _ptr(y), _stream(stream)))


def moe_combine_tokens(h: Handle, begin: int, end: int, y, w, out, stream=None) -> None:
    _check("moe_combine_tokens", load_library().moe_combine_tokens(
        h.ptr, int(begin), int(end), _ptr(y), _ptr(w), _ptr(out), _stream(stream)))


def moe_dispatch_allgather(h: Handle, x, w, gathered_x, gathered_scale, recv_x, recv_scale,
                           meta: dict, stream=None) -> None:
    m = moe_recv_meta_t(*(_ptr(meta[n]) for n in (
        "local_expert", "src_rank", "src_token", "slot", "weight")))
    _check("moe_dispatch_allgather", load_library().moe_dispatch_allgather(
        h.ptr, _ptr(x), _ptr(w), _ptr(gathered_x), _ptr(gathered_scale), _ptr(recv_x),
        _ptr(recv_scale), ctypes.byref(m), _stream(stream)))


def moe_expert_standin(h: Handle, recv_x, recv_scale, expert_scale, y, stream=None) -> None:
    _check("moe_expert_standin", load_library().moe_expert_standin(
        h.ptr, _ptr(recv_x), _ptr(recv_scale), _ptr(expert_scale), _ptr(y), _stream(stream)))


def moe_combine(h: Handle, y, w, out, stream=None) -> None:
    _check("moe_combine", load_library().moe_combine(
        h.ptr, _ptr(y), _ptr(w), _ptr(out), _stream(stream)))


def moe_read_status(h: Handle, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check("moe_read_status", load_library().moe_read_status(
        h.ptr, ctypes.byref(flags), _stream(stream)))
    return int(flags.value)


def moe_dispatch_layout_noalloc(cfg: moe_config_t, ids, out: dict, stream=None) -> None:
    """Layout + inverse permutation into caller tensors (int32, sized as in
    moe_get_layout's views), with no device allocation by the library. For
    callers that cannot allocate (graph capture, fixed-pool runtimes); the
    first call on a device must precede any stream capture; overlapping calls
    race on the library's static scratch."""
    v = moe_layout_view_t(*(_ptr(out[n]) for n, _ in moe_layout_view_t._fields_))
    _check("moe_dispatch_layout_noalloc", load_library().moe_dispatch_layout_noalloc(
        ctypes.byref(cfg), _ptr(ids), ctypes.byref(v), _stream(stream)))


def _host_ptr(t) -> int:
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def moe_copy_h2d_async(dst, src_host, stream=None) -> None:
    """Stream-ordered copy of a (pinned) host tensor into a device tensor."""
    n = src_host.numel() * src_host.element_size()
    if n != dst.numel() * dst.element_size():
        raise ValueError("size mismatch")
    _check("moe_copy_h2d_async", load_library().moe_copy_h2d_async(
        _ptr(dst), _host_ptr(src_host), n, _stream(stream)))


def moe_copy_d2h_async(dst_host, src, stream=None) -> None:
    """Stream-ordered copy of a device tensor into a (pinned) host tensor."""
    n = src.numel() * src.element_size()
    if n != dst_host.numel() * dst_host.element_size():
        raise ValueError("size mismatch")
    _check("moe_copy_d2h_async", load_library().moe_copy_d2h_async(
        _host_ptr(dst_host), _ptr(src), n, _stream(stream)))


def moe_error_string(code: int) -> str:
    return load_library().moe_error_string(code).decode()


def moe_debug_bounds() -> bool:
    """True if the loaded library checks every computed row index on the device."""
    return bool(load_library().moe_debug_bounds())
