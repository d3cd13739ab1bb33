"""CPU oracle for the MoE expert-parallel dispatch/combine path.

TEST INFRASTRUCTURE ONLY. The product library never imports, links or calls
anything here; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do. The arithmetic lives in ``moe_oracle.c`` (plain C,
explicit loops, IEEE float without contraction); this module compiles it with
gcc on first use and marshals numpy arrays through ctypes.

Sources of each definition (page title, section):
  * route: "Efficient and portable MoE communication" (pplx-kernels blog),
    introduction -- router top-k and weighted sum; "Expert Parallel: MoE
    Token ...", "A Top-2 routing example" -- [num_tokens, top_k] router output.
  * layout: "Expert Parallel: MoE Token ...", "Why count and permute before
    dispatch" (owner, send_count, prefix sum, destination-contiguous writes,
    bijection) and "All-to-All-v" (count matrix C_ij); "[Infra-10] All-to-All
    Optimization", 8.1 (capacity and dropping).
  * dispatch payload: "Expert Parallel ...", payload schema; "[Infra-10]", 2.1
    and 4.1 (quantisation scale metadata, FP8 on the wire).
  * combine: "Expert Parallel ...", "Combine is not simply sending results
    back"; pplx blog, "Combine".

Parity status: every function is pinned by tests/test_oracle_pins.py except the
route weights' last fp32 bit, whose only pins are the library softmax and the
renormalisation identity (no page prints a top-k result for given logits).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared object (gcc, -O2, no contraction)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
        "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oref_bf16_from_f32.restype = ctypes.c_uint16
        lib.oref_bf16_from_f32.argtypes = [ctypes.c_float]
        lib.oref_f32_from_bf16.restype = ctypes.c_float
        lib.oref_f32_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oref_e4m3_value.restype = ctypes.c_double
        lib.oref_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oref_e4m3_from_f32.restype = ctypes.c_uint8
        lib.oref_e4m3_from_f32.argtypes = [ctypes.c_float]
        lib.oref_route_topk.restype = None
        lib.oref_route_topk.argtypes = [_i64, _int, _int, _f32p, _i32p, _f32p]
        lib.oref_layout_flat.restype = _i64
        lib.oref_layout_flat.argtypes = [_int, _i64, _int, _int, _i64, _i32p] + [_i32p] * 11
        lib.oref_dispatch_bf16.restype = None
        lib.oref_dispatch_bf16.argtypes = [_int, _i64, _int, _int, _i64, _i32p, _i32p,
                                           _u16p, _f32p, _u16p, _i32p, _i32p, _i32p,
                                           _i32p, _f32p]
        lib.oref_dispatch_fp8.restype = None
        lib.oref_dispatch_fp8.argtypes = [_int, _i64, _int, _int, _i64, _i32p, _i32p,
                                          _u16p, _f32p, _u8p, _f32p, _i32p, _i32p,
                                          _i32p, _i32p, _f32p]
        lib.oref_quantize_row_fp8.restype = None
        lib.oref_quantize_row_fp8.argtypes = [_i64, _u16p, _u8p, _f32p]
        lib.oref_expert_scale_bf16.restype = None
        lib.oref_expert_scale_bf16.argtypes = [_int, _i64, _i32p, _f32p, _u16p, _u16p]
        lib.oref_expert_dequant_fp8.restype = None
        lib.oref_expert_dequant_fp8.argtypes = [_i64, _i64, _u8p, _f32p, _u16p]
        lib.oref_combine.restype = None
        lib.oref_combine.argtypes = [_i64, _int, _i64, _i32p, _f32p, _u16p, _u16p]
        lib.oref_combine_token.restype = None
        lib.oref_combine_token.argtypes = [_int, _i64, _i32p, _f32p, _u16p, _u16p]
        _lib = lib
        return lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# token-range shards (marshalling only: the C functions run unchanged)
# --------------------------------------------------------------------------
def _ranges(n: int, threads: int):
    """[a, b) token ranges of about n / threads tokens each."""
    threads = max(1, min(int(threads), n))
    b = [n * i // threads for i in range(threads + 1)]
    return [(b[i], b[i + 1]) for i in range(threads) if b[i + 1] > b[i]]


def _run(jobs):
    """Runs the jobs (calls into the C library, which release the GIL) on one
    thread each; a single job runs inline."""
    if len(jobs) <= 1:
        for j in jobs:
            j()
        return
    with ThreadPoolExecutor(len(jobs)) as ex:
        for f in [ex.submit(j) for j in jobs]:
            f.result()


def _shard_inv(inv: np.ndarray, k: int, a: int, b: int) -> np.ndarray:
    """inv with every assignment outside tokens [a, b) marked -1, so that an
    unchanged dispatch call writes exactly the rows of those tokens."""
    out = np.full_like(inv, -1)
    out[a * k:b * k] = inv[a * k:b * k]
    return out


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def bf16_from_f32(v: float) -> int:
    return int(_load().oref_bf16_from_f32(float(v)))


def f32_from_bf16(h: int) -> float:
    return float(_load().oref_f32_from_bf16(int(h)))


def e4m3_value(code: int) -> float:
    return float(_load().oref_e4m3_value(int(code)))


def e4m3_from_f32(v: float) -> int:
    return int(_load().oref_e4m3_from_f32(float(v)))


# --------------------------------------------------------------------------
# path steps
# --------------------------------------------------------------------------
def route_topk(logits: np.ndarray, k: int, threads: int = 1):
    """Top-k ids (descending logit, ties to the lower expert) and the softmax of
    the chosen logits (double, rounded to fp32). threads > 1 runs the same C
    function on token ranges concurrently (tokens are independent)."""
    z = _c(logits, np.float32)
    T, E = z.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    lib = _load()
    _run([lambda a=a, b=b: lib.oref_route_topk(b - a, E, k, z[a:b], ids[a:b], w[a:b])
          for a, b in _ranges(T, threads)])
    return ids, w


def layout(P: int, Tr: int, E: int, k: int, ids: np.ndarray, cap: int = 0) -> dict:
    """Counts, offsets, count matrix and receive row of every assignment."""
    ids = _c(ids, np.int32).reshape(-1)
    Na = P * Tr * k
    assert ids.size == Na
    out = dict(
        n_raw=np.empty(E, np.int32), n_kept=np.empty(E, np.int32),
        expert_offset=np.empty(E + 1, np.int32), cnt=np.empty((P, E), np.int32),
        kept_cnt=np.empty((P, E), np.int32), C=np.empty((P, P), np.int32),
        send_offset=np.empty((P, P), np.int32), recv_offset=np.empty((P, E), np.int32),
        rank_base=np.empty(P + 1, np.int32), inv=np.empty(Na, np.int32),
        totals=np.empty(3, np.int32))
    bad = _load().oref_layout_flat(
        P, Tr, E, k, cap, ids, out["n_raw"], out["n_kept"], out["expert_offset"],
        out["cnt"], out["kept_cnt"], out["C"], out["send_offset"], out["recv_offset"],
        out["rank_base"], out["inv"], out["totals"])
    out["bad_ids"] = int(bad)
    return out


def _meta(rows):
    return dict(local_expert=np.full(rows, -7, np.int32), src_rank=np.full(rows, -7, np.int32),
                src_token=np.full(rows, -7, np.int32), slot=np.full(rows, -7, np.int32),
                weight=np.full(rows, np.nan, np.float32))


def dispatch_bf16(P, Tr, E, k, x_bits: np.ndarray, w: np.ndarray, ids: np.ndarray,
                  inv: np.ndarray, rows: int, threads: int = 1):
    """Receive rows [rows, H] (bf16 bits) and metadata, from x bits [T, H].
    threads > 1: each thread runs the same C function with the assignments of
    its token range only (the others marked -1); the rows they write are
    disjoint."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    recv = np.zeros((rows, H), np.uint16)
    m = _meta(rows)
    ids_f, inv_f, w_f = (_c(ids, np.int32).reshape(-1), _c(inv, np.int32).reshape(-1),
                         _c(w, np.float32).reshape(-1))
    lib = _load()
    parts = _ranges(T, threads)

    def job(a, b):
        inv_s = inv_f if len(parts) == 1 else _shard_inv(inv_f, k, a, b)
        lib.oref_dispatch_bf16(P, Tr, E, k, H, ids_f, inv_s, x_bits, w_f, recv,
                               m["local_expert"], m["src_rank"], m["src_token"], m["slot"],
                               m["weight"])
    _run([lambda a=a, b=b: job(a, b) for a, b in parts])
    return recv, m


def dispatch_fp8(P, Tr, E, k, x_bits, w, ids, inv, rows: int, threads: int = 1):
    """FP8 receive rows [rows, H] (e4m3 codes), scales [rows, H/128] and
    metadata; threads as in dispatch_bf16."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    recv = np.zeros((rows, H), np.uint8)
    sc = np.zeros((rows, H // 128), np.float32)
    m = _meta(rows)
    ids_f, inv_f, w_f = (_c(ids, np.int32).reshape(-1), _c(inv, np.int32).reshape(-1),
                         _c(w, np.float32).reshape(-1))
    lib = _load()
    parts = _ranges(T, threads)

    def job(a, b):
        inv_s = inv_f if len(parts) == 1 else _shard_inv(inv_f, k, a, b)
        lib.oref_dispatch_fp8(P, Tr, E, k, H, ids_f, inv_s, x_bits, w_f, recv, sc,
                              m["local_expert"], m["src_rank"], m["src_token"], m["slot"],
                              m["weight"])
    _run([lambda a=a, b=b: job(a, b) for a, b in parts])
    return recv, sc, m


def quantize_row_fp8(x_row_bits: np.ndarray):
    x_row_bits = _c(x_row_bits, np.uint16)
    H = x_row_bits.shape[0]
    q = np.empty(H, np.uint8)
    sc = np.empty(H // 128, np.float32)
    _load().oref_quantize_row_fp8(H, x_row_bits, q, sc)
    return q, sc


def expert_scale_bf16(E, expert_offset, c, recv_bits):
    recv_bits = _c(recv_bits, np.uint16)
    y = np.zeros_like(recv_bits)
    _load().oref_expert_scale_bf16(E, recv_bits.shape[1], _c(expert_offset, np.int32),
                                   _c(c, np.float32), recv_bits, y)
    return y


def expert_dequant_fp8(recv_q, recv_scale, threads: int = 1):
    """threads > 1: the same C function on row ranges (rows are independent)."""
    recv_q = _c(recv_q, np.uint8)
    rows, H = recv_q.shape
    y = np.zeros((rows, H), np.uint16)
    s = _c(recv_scale, np.float32)
    lib = _load()
    _run([lambda a=a, b=b: lib.oref_expert_dequant_fp8(b - a, H, recv_q[a:b], s[a:b], y[a:b])
          for a, b in _ranges(rows, threads)])
    return y


def combine(inv: np.ndarray, w: np.ndarray, y_bits: np.ndarray, T: int, k: int,
            threads: int = 1):
    """threads > 1: the same C function on token ranges (each output token
    reads only its own slots)."""
    y_bits = _c(y_bits, np.uint16)
    H = y_bits.shape[1]
    out = np.empty((T, H), np.uint16)
    inv_f, w_f = _c(inv, np.int32).reshape(-1), _c(w, np.float32).reshape(-1)
    lib = _load()
    _run([lambda a=a, b=b: lib.oref_combine(b - a, k, H, inv_f[a * k:b * k], w_f[a * k:b * k],
                                            y_bits, out[a:b])
          for a, b in _ranges(T, threads)])
    return out


def combine_token(inv_g: np.ndarray, w_g: np.ndarray, y_bits: np.ndarray):
    """One token's combine; y_bits holds all receive rows (indexed by inv_g)."""
    y_bits = _c(y_bits, np.uint16)
    H = y_bits.shape[1]
    k = int(np.asarray(inv_g).size)
    out = np.empty(H, np.uint16)
    _load().oref_combine_token(k, H, _c(inv_g, np.int32), _c(w_g, np.float32), y_bits, out)
    return out
