"""The five synthetic workloads of the VeriCache draft-then-verify round.

Each workload fixes attention shapes, per-request context lengths, the compression
mode of every request, the draft length L, the vocabulary and the planted match
probability. The shapes follow the model classes the VeriCache summary evaluates
(Llama-, Qwen- and Mistral-class attention, long contexts, 25-40-token drafts;
"VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", sections
"Core algorithm", "Extended verification period (P2)" and "Experimental results").
This module holds sizes only: no arithmetic of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List

import numpy as np

DROP = "drop"
QUANT = "quant"


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    ctx: List[int]
    mode: List[str]
    keep: List[int]          # token drop: kept rows k (0 for quant requests)
    recent: List[int]        # token drop: recent window R always kept
    bits: int                # quant: 2 or 4
    residual_min: int        # quant: at least this many trailing tokens stay bf16
    L: List[int]             # draft length per request
    V: int                   # vocabulary
    p: List[float]           # planted match probability per request
    on_host: List[bool]      # full KV held in pinned host memory
    rounds: int = 1
    seed: int = 0
    note: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def L_max(self) -> int:
        return max(self.L)

    def request_indices(self, mode: str) -> List[int]:
        return [b for b in range(self.B) if self.mode[b] == mode]


def _uniform(B, v):
    return [v] * B


def tiny() -> Workload:
    """Single layer, batch 1, 8/2 heads, d 64, context 1024, keep 256 (no recent window), L 8."""
    B = 1
    return Workload("tiny_drop_b1_ctx1k", B, 8, 2, 64, _uniform(B, 1024), _uniform(B, DROP),
                    _uniform(B, 256), _uniform(B, 0), 2, 128, _uniform(B, 8), 1000,
                    _uniform(B, 0.9), _uniform(B, False))


def llama8b_drop() -> Workload:
    """Llama-3-8B attention shape, batch 8, context 32768, keep 8192 = last 512 + top 7680, L 32."""
    B = 8
    return Workload("llama8b_drop4x_b8_ctx32k", B, 32, 8, 128, _uniform(B, 32768), _uniform(B, DROP),
                    _uniform(B, 8192), _uniform(B, 512), 2, 128, _uniform(B, 32), 128256,
                    _uniform(B, 0.95), _uniform(B, False))


def qwen32b_quant2() -> Workload:
    """Qwen-32B-like shape, batch 16, 40/8 heads, context 65536, 2-bit keys and values, L 25."""
    B = 16
    return Workload("qwen32b_kivi2_b16_ctx64k", B, 40, 8, 128, _uniform(B, 65536), _uniform(B, QUANT),
                    _uniform(B, 0), _uniform(B, 0), 2, 128, _uniform(B, 25), 152064,
                    _uniform(B, 0.93), _uniform(B, False))


def llama70b_offload4() -> Workload:
    """Llama-70B long-context offload: batch 4, 64/8 heads, context 131072, 4-bit, full KV on host, L 40.

    Two requests draft while the other two stage their full KV and verify, then the roles swap.
    """
    B = 4
    return Workload("llama70b_kivi4_offload_b4_ctx128k", B, 64, 8, 128, _uniform(B, 131072),
                    _uniform(B, QUANT), _uniform(B, 0), _uniform(B, 0), 4, 128, _uniform(B, 40),
                    128256, _uniform(B, 0.95), _uniform(B, True))


def mixed_serving(seed: int = 0) -> Workload:
    """32 requests, 32/8 heads, contexts log-uniform in [8K, 256K], half drop-4x and half 2-bit,
    L uniform in [25, 40], half the full caches on the host, match probability uniform in
    [0.85, 0.98], 20 rounds. Request b uses token drop when b is even and quantization when b is
    odd; its full KV sits on the host when (b // 2) is odd, so each mode has both residencies."""
    B = 32
    rng = np.random.default_rng(1000 + seed)
    lo, hi = math.log(8192), math.log(262144)
    ctx = [int(round(math.exp(x))) for x in rng.uniform(lo, hi, size=B)]
    L = [int(x) for x in rng.integers(25, 41, size=B)]
    p = [float(x) for x in rng.uniform(0.85, 0.98, size=B)]
    mode = [DROP if b % 2 == 0 else QUANT for b in range(B)]
    keep = [c // 4 if m == DROP else 0 for c, m in zip(ctx, mode)]
    recent = [512 if m == DROP else 0 for m in mode]
    on_host = [(b // 2) % 2 == 1 for b in range(B)]
    return Workload("mixed_staggered_32req_ctx8k_256k", B, 32, 8, 128, ctx, mode, keep, recent, 2, 128,
                    L, 128256, p, on_host, rounds=20, seed=seed)


def subset(w: Workload, pick: List[int], name: str | None = None) -> Workload:
    """The requests `pick` of w, in that order, as a workload of their own (same shapes)."""
    sel = lambda xs: [xs[b] for b in pick]
    return Workload(name or (w.name + f"_sub{len(pick)}"), len(pick), w.Hq, w.Hkv, w.d, sel(w.ctx), sel(w.mode),
                    sel(w.keep), sel(w.recent), w.bits, w.residual_min, sel(w.L), w.V, sel(w.p), sel(w.on_host),
                    w.rounds, w.seed)


ALL = [tiny, llama8b_drop, qwen32b_quant2, llama70b_offload4, mixed_serving]


def by_index(i: int) -> Workload:
    return ALL[i]()


def scaled(w: Workload, ctx_div: int = 1, batch: int | None = None, vocab: int | None = None,
           L: int | None = None) -> Workload:
    """A smaller copy of a workload with the same head shape and compression mode, for parity
    cases the oracle finishes in seconds. Context, keep and recent scale down together."""
    B = batch if batch is not None else w.B
    pick = list(range(B))
    ctx = [max(1, w.ctx[b % w.B] // ctx_div) for b in pick]
    keep = [max(0, w.keep[b % w.B] // ctx_div) for b in pick]
    recent = [min(w.recent[b % w.B] // ctx_div, k) for b, k in zip(pick, keep)]
    Ls = [L if L is not None else w.L[b % w.B] for b in pick]
    return Workload(w.name + f"_div{ctx_div}_b{B}", B, w.Hq, w.Hkv, w.d, ctx,
                    [w.mode[b % w.B] for b in pick], keep, recent, w.bits, w.residual_min, Ls,
                    vocab if vocab is not None else w.V, [w.p[b % w.B] for b in pick],
                    [w.on_host[b % w.B] for b in pick], w.rounds, w.seed)
