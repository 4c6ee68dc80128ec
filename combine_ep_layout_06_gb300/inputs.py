"""Seeded synthetic inputs for MoE token dispatch / combine.

This module only draws random inputs.  It holds none of the method's
arithmetic (no routing layout, no copy, no quantisation, no reduction), so
that the CPU oracle and the CUDA path can both consume it without sharing
any code that computes a result.

Workloads (shapes and distributions of the MoE expert-parallel workloads the
MORI-EP "Communication APIs" page targets with ``EpDispatchCombineOp``):

============  ==  ===  ==  =====  ====  ======================================
name          W   E    k   T      H     routing / payload
============  ==  ===  ==  =====  ====  ======================================
tiny          2   8    2   128    256   uniform distinct top-k, N(0,1)
dsv3          8   256  8   4096   7168  uniform distinct top-k, N(0,1)
dsv3_fp8_zipf 8   256  8   4096   7168  Zipf(1.2) over a random expert
                                        permutation, fused FP8 E4M3 dispatch
ll_decode     16  256  8   128    7168  uniform, split send/recv streams
mixtral       8   8    2   16384  4096  uniform over experts 0..5 only, so
                                        ranks 6 and 7 receive nothing; N(0,2)
============  ==  ===  ==  =====  ====  ======================================

Draw order for every workload (numpy ``default_rng(PCG64(seed))``):
x (float32 normal, then a round-to-nearest-even cast to bf16 by torch's CPU
cast), then the routing keys, then the weight logits.  Weights are a float32
softmax over the k chosen experts, so each row sums to 1 within fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    world_size: int          # W logical EP ranks
    num_experts: int         # E
    topk: int                # k
    max_tokens_per_rank: int  # T
    hidden: int              # H
    routing: str = "uniform"  # "uniform" | "zipf" | "restricted"
    zipf_s: float = 1.2
    restrict_experts: int = 0  # routing uses experts [0, restrict_experts)
    x_std: float = 1.0
    fp8: bool = False        # fused FP8 E4M3 dispatch payload
    split: bool = False      # split send/recv on two streams
    seed: int = 0

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.world_size

    def scaled(self, tokens: int, hidden: Optional[int] = None) -> "Workload":
        """Same routing recipe at a smaller token count (and hidden size)."""
        return dataclasses.replace(
            self, max_tokens_per_rank=tokens,
            hidden=self.hidden if hidden is None else hidden)


WORKLOADS = {
    "tiny": Workload("tiny", 2, 8, 2, 128, 256),
    "dsv3": Workload("dsv3", 8, 256, 8, 4096, 7168),
    "dsv3_fp8_zipf": Workload("dsv3_fp8_zipf", 8, 256, 8, 4096, 7168,
                              routing="zipf", fp8=True),
    "ll_decode": Workload("ll_decode", 16, 256, 8, 128, 7168, split=True),
    "mixtral": Workload("mixtral", 8, 8, 2, 16384, 4096,
                        routing="restricted", restrict_experts=6,
                        x_std=math.sqrt(2.0)),
}


@dataclasses.dataclass
class Inputs:
    wl: Workload
    x_bits: np.ndarray       # uint16 [W][T][H], bf16 bit patterns
    weights: np.ndarray      # float32 [W][T][k]
    indices: np.ndarray      # int32 [W][T][k], global expert ids
    num_tokens: np.ndarray   # int32 [W], tokens present on each source rank


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values, via torch's CPU cast (RNE)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw_routing(rng: np.random.Generator, wl: Workload, n: int) -> np.ndarray:
    """Distinct top-k expert ids for n tokens, int32 [n][k]."""
    E, k = wl.num_experts, wl.topk
    if wl.routing == "uniform":
        keys = rng.random((n, E))
        sel = np.argsort(keys, axis=1, kind="stable")[:, :k]
    elif wl.routing == "restricted":
        Er = wl.restrict_experts
        keys = rng.random((n, Er))
        sel = np.argsort(keys, axis=1, kind="stable")[:, :k]
    elif wl.routing == "zipf":
        perm = rng.permutation(E)
        p = (np.arange(E, dtype=np.float64) + 1.0) ** (-wl.zipf_s)
        p /= p.sum()
        logp = np.empty(E)
        logp[perm] = np.log(p)          # expert perm[i] has popularity rank i
        g = rng.gumbel(size=(n, E))      # Gumbel-top-k == sampling w/o replacement
        sel = np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k]
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    return sel.astype(np.int32)


def draw_weights(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """Softmax (float32) of N(0,1) logits over the k chosen experts."""
    logits = rng.standard_normal((n, k)).astype(np.float32)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m, dtype=np.float32)
    return (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def make_inputs(wl: Workload, num_tokens: Optional[Sequence[int]] = None,
                seed: Optional[int] = None) -> Inputs:
    """Draw one batch for ``wl``.  ``num_tokens`` (per source rank, each
    <= T) defaults to a full batch; the rows of absent tokens still hold
    drawn data but take no part in the method."""
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    rng = np.random.default_rng(np.random.PCG64(wl.seed if seed is None else seed))
    n = W * T
    x = np.empty((n, H), dtype=np.uint16)
    rows = max(1, (1 << 26) // max(H, 1))   # draw in ~256 MB float32 slabs
    for r0 in range(0, n, rows):
        r1 = min(n, r0 + rows)
        xf = rng.standard_normal((r1 - r0, H), dtype=np.float32)
        if wl.x_std != 1.0:
            xf *= np.float32(wl.x_std)
        x[r0:r1] = _bf16_bits_from_f32(xf)
    idx = draw_routing(rng, wl, n)
    w = draw_weights(rng, n, k)
    if num_tokens is None:
        nt = np.full(W, T, dtype=np.int32)
    else:
        nt = np.asarray(num_tokens, dtype=np.int32)
        if nt.shape != (W,) or (nt < 0).any() or (nt > T).any():
            raise ValueError("num_tokens must be W values in [0, T]")
    return Inputs(wl, x.reshape(W, T, H), w.reshape(W, T, k),
                  idx.reshape(W, T, k), nt)


def ragged_num_tokens(wl: Workload, seed: int = 1) -> np.ndarray:
    """A ragged per-rank token count including an empty and a full rank."""
    rng = np.random.default_rng(seed)
    T, W = wl.max_tokens_per_rank, wl.world_size
    nt = rng.integers(0, T + 1, size=W).astype(np.int32)
    nt[0] = T
    if W > 1:
        nt[W - 1] = 0
    return nt


def draw_fp8_payload(wl: Workload, seed: int = 7):
    """A pre-quantised FP8 payload for the pass-through dispatch: random
    E4M3 codes (both NaN patterns excluded) [W][T][H] and positive fp32
    block scales [W][T][H/128] (log-uniform over 2^-20 .. 2^4)."""
    W, T, H = wl.world_size, wl.max_tokens_per_rank, wl.hidden
    rng = np.random.default_rng(np.random.PCG64(seed))
    codes = rng.integers(0, 254, size=(W, T, H)).astype(np.uint8)
    codes[codes >= 0x7F] += 1          # 0..126, 128..254: skips 0x7F and 0xFF
    scales = np.exp2(rng.uniform(-20.0, 4.0, size=(W, T, H // 128))).astype(np.float32)
    return codes, scales
