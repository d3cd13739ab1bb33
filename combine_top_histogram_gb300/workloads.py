"""Seeded synthetic inputs for the MoE dispatch/combine path.

This module only draws inputs; it holds none of the path's arithmetic (no
top-k, no counting, no packing, no combine). Both the CPU oracle and the CUDA
library are fed from here, so the two sides always see identical bytes.

The five workloads follow the pages' benchmark dimensions ("[Infra-10]
All-to-All Optimization", 11.3: token count, hidden size, top-k, uniform vs
Zipf hot spots, BF16 vs low precision, prefill vs decode) and the worked
example of "Expert Parallel: MoE Token ...", "A Top-2 routing example". No
public dataset or routing trace is involved; every array is drawn from
``numpy.random.default_rng(seed)`` in the fixed order documented per field.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

MOE_BF16 = 0
MOE_FP8_E4M3 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int            # virtual EP ranks
    Tr: int           # tokens per rank
    E: int            # experts
    k: int            # top-k
    H: int            # hidden size
    dispatch_dtype: int
    routing: str      # "fixed" | "logits" | "uniform" | "zipf"
    expert: str       # "identity" | "scale" | "dequant"
    cap: int = 0      # per-expert capacity, 0 = unlimited
    seed: int = 0
    zipf_s: float = 1.2

    @property
    def T(self) -> int:
        return self.P * self.Tr

    @property
    def Na(self) -> int:
        return self.T * self.k

    @property
    def L(self) -> int:
        return self.E // self.P

    @property
    def rows_max(self) -> int:
        """Receive rows the caller must provide: N_a, or E*cap when that is smaller."""
        if self.cap > 0:
            return min(self.Na, self.E * self.cap)
        return self.Na

    def scaled(self, name: str, Tr: int, H: Optional[int] = None, cap: Optional[int] = None):
        return dataclasses.replace(self, name=name, Tr=Tr, H=self.H if H is None else H,
                                   cap=self.cap if cap is None else cap)


def prefill_capacity(T_total: int, k: int, E: int, factor: float = 1.25) -> int:
    """ceil(factor * T_total * k / E): the prefill workload's per-expert limit."""
    return int(math.ceil(factor * T_total * k / E))


# The worked example's routing ("Expert Parallel: MoE Token ...", "A Top-2
# routing example"): 4 ranks x 2 tokens, 8 experts, top-2.
WORKED_ROUTING = np.array([[1, 6], [4, 7], [1, 5], [2, 4], [0, 7], [3, 6], [2, 5], [0, 3]],
                          dtype=np.int32)

WORKED = Workload("worked_p4_t8_e8_k2_h128_bf16", 4, 2, 8, 2, 128, MOE_BF16, "fixed",
                  "identity", seed=1)
DECODE = Workload("decode_p8x128_e256_k8_h7168_bf16", 8, 128, 256, 8, 7168, MOE_BF16,
                  "logits", "scale", seed=2)
UNIFORM_FP8 = Workload("uniform_p8x2048_e64_k2_h7168_fp8", 8, 2048, 64, 2, 7168,
                       MOE_FP8_E4M3, "uniform", "dequant", seed=3)
SKEWED = Workload("zipf1.2_p8x4096_e8_k2_h4096_bf16", 8, 4096, 8, 2, 4096, MOE_BF16,
                  "zipf", "identity", seed=4)
PREFILL = Workload("prefill_p32x4096_e256_k8_h7168_fp8_cap5120", 32, 4096, 256, 8, 7168,
                   MOE_FP8_E4M3, "logits", "dequant", cap=prefill_capacity(32 * 4096, 8, 256),
                   seed=5)

CONFIGS = {"worked": WORKED, "decode": DECODE, "uniform_fp8": UNIFORM_FP8,
           "skewed": SKEWED, "prefill": PREFILL}


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (round-to-nearest-even, by torch's cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw_hidden(rng: np.random.Generator, T: int, H: int, rows_per_draw: int = 4096) -> np.ndarray:
    """x ~ N(0,1) in fp32, rounded to bf16; drawn in blocks of rows to bound memory."""
    out = np.empty((T, H), np.uint16)
    for r0 in range(0, T, rows_per_draw):
        r1 = min(T, r0 + rows_per_draw)
        out[r0:r1] = _bf16_bits_from_f32(rng.standard_normal((r1 - r0, H), dtype=np.float32))
    return out


def _gumbel_topk_draws(rng: np.random.Generator, logp: np.ndarray, T: int, k: int) -> np.ndarray:
    """k draws without replacement per token, in draw order (Gumbel-top-k)."""
    E = logp.shape[0]
    u = rng.random((T, E))
    keys = logp[None, :] - np.log(-np.log(u))
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _softmax_weights(rng: np.random.Generator, T: int, k: int) -> np.ndarray:
    """Weights for externally drawn ids: softmax of k N(0,1) logits (fp64 -> fp32)."""
    z = rng.standard_normal((T, k))
    z = z - z.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return (ez / ez.sum(axis=1, keepdims=True)).astype(np.float32)


@dataclasses.dataclass
class Inputs:
    wl: Workload
    x: np.ndarray                       # uint16 bf16 bits [T, H]
    logits: Optional[np.ndarray]        # fp32 [T, E] when routing == "logits"
    ids: Optional[np.ndarray]           # int32 [T, k] when routing is given
    w: Optional[np.ndarray]             # fp32 [T, k] when routing is given
    expert_scale: Optional[np.ndarray]  # fp32 [E] for the "scale" expert


def make_inputs(wl: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw order: x, then routing (logits, or ids then weights), then expert scales."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    x = draw_hidden(rng, wl.T, wl.H)
    logits = ids = w = c = None
    if wl.routing == "fixed":
        assert (wl.P, wl.Tr, wl.E, wl.k) == (4, 2, 8, 2)
        ids = WORKED_ROUTING.copy()
        w = np.tile(np.array([0.6, 0.4], np.float32), (wl.T, 1))
    elif wl.routing == "logits":
        logits = rng.standard_normal((wl.T, wl.E), dtype=np.float32)
    elif wl.routing == "uniform":
        ids = _gumbel_topk_draws(rng, np.zeros(wl.E), wl.T, wl.k)
        w = _softmax_weights(rng, wl.T, wl.k)
    elif wl.routing == "zipf":
        p = (np.arange(wl.E) + 1.0) ** (-wl.zipf_s)
        ids = _gumbel_topk_draws(rng, np.log(p / p.sum()), wl.T, wl.k)
        w = _softmax_weights(rng, wl.T, wl.k)
    else:
        raise ValueError(wl.routing)
    if wl.expert == "scale":
        c = (rng.random(wl.E, dtype=np.float32) + np.float32(0.5)).astype(np.float32)
    return Inputs(wl, x, logits, ids, w, c)


def mask_random_slots(ids: np.ndarray, frac: float, seed: int) -> np.ndarray:
    """Marks a random fraction of slots as padding (-1)."""
    rng = np.random.default_rng(seed)
    out = ids.copy()
    out[rng.random(ids.shape) < frac] = -1
    return out
