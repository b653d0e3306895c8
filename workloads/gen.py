"""Seeded synthetic inputs for one VeriCache round, shared by the oracle tests and the CUDA path.

The generator draws every tensor from its own torch.Generator, seeded from
(workload seed, round, request, tensor kind), so a request's tensors do not depend on the
device or on the other requests. It holds no arithmetic of the method: the planted-argmax
logits are an input recipe (base N(0,1); with probability p the drafted token is made the
row's unique maximum, otherwise it is pushed below the row minimum when it happens to be the
argmax), and draws for it are made here, not by the code under test.

Per request b of a round:
  k_full, v_full  bf16 [Hkv][ctx][d]   ~ N(0,1)
  importance      fp32 [ctx]           ~ U[0,1)        (token-drop requests)
  q               bf16 [L][Hq][d]      ~ N(0,1)        query of draft step s = verify row s
  k_new, v_new    bf16 [L][Hkv][d]     ~ N(0,1)        the drafted tokens' own K/V
For the batch:
  draft           int32 [B][L_max]     uniform in [0, V); 0 beyond L_b
  logits          fp32 [B][L_max+1][V] planted as above for rows < L_b
  L               int32 [B]
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

import torch

from .configs import Workload, DROP

(KIND_K, KIND_V, KIND_IMP, KIND_Q, KIND_KNEW, KIND_VNEW, KIND_DRAFT, KIND_LOGITS, KIND_PLANT, KIND_APPK, KIND_APPV,
 KIND_QOBS) = range(12)


def _gen(w: Workload, rnd: int, b: int, kind: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 1_000_003 + rnd) * 10_007 + b) * 101 + kind)
    return g


def randn_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class RequestInputs:
    k_full: torch.Tensor
    v_full: torch.Tensor
    importance: torch.Tensor | None
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor


def full_kv(w: Workload, b: int, device="cpu"):
    """The request's full cache: (k, v), each bf16 [Hkv][ctx][d]. Independent of the round."""
    shape = (w.Hkv, w.ctx[b], w.d)
    return (randn_bf16(shape, _gen(w, 0, b, KIND_K, device), device),
            randn_bf16(shape, _gen(w, 0, b, KIND_V, device), device))


def importance(w: Workload, b: int, device="cpu", n: int | None = None) -> torch.Tensor:
    """fp32 [n] ~ U[0,1) (n defaults to the context; a longer array serves a context that grows)."""
    g = _gen(w, 0, b, KIND_IMP, device)
    return torch.rand((w.ctx[b] if n is None else n,), generator=g, device=device, dtype=torch.float32)


def observation_queries(w: Workload, b: int, window: int, device="cpu") -> torch.Tensor:
    """bf16 [window][Hq][d] ~ N(0,1): queries of the request's last `window` context tokens."""
    return randn_bf16((window, w.Hq, w.d), _gen(w, 0, b, KIND_QOBS, device), device)


def appended_rows(w: Workload, rnd: int, b: int, n: int, device="cpu"):
    """(k, v) bf16 [n][Hkv][d] ~ N(0,1): rows a request's cache gains after round rnd."""
    shape = (n, w.Hkv, w.d)
    return (randn_bf16(shape, _gen(w, rnd, b, KIND_APPK, device), device),
            randn_bf16(shape, _gen(w, rnd, b, KIND_APPV, device), device))


def round_queries(w: Workload, rnd: int, b: int, device="cpu"):
    """(q [L][Hq][d], k_new [L][Hkv][d], v_new [L][Hkv][d]) for request b in round rnd."""
    L = w.L[b]
    q = randn_bf16((L, w.Hq, w.d), _gen(w, rnd, b, KIND_Q, device), device)
    kn = randn_bf16((L, w.Hkv, w.d), _gen(w, rnd, b, KIND_KNEW, device), device)
    vn = randn_bf16((L, w.Hkv, w.d), _gen(w, rnd, b, KIND_VNEW, device), device)
    return q, kn, vn


def request(w: Workload, rnd: int, b: int, device="cpu") -> RequestInputs:
    k, v = full_kv(w, b, device)
    imp = importance(w, b, device) if w.mode[b] == DROP else None
    q, kn, vn = round_queries(w, rnd, b, device)
    return RequestInputs(k, v, imp, q, kn, vn)


def request_logits(w: Workload, rnd: int, b: int, device="cpu", vocab: int | None = None, out=None):
    """Request b's row of drafts_and_logits: (draft int32 [L_max], logits fp32 [L_max+1][V]), written
    into `out` = (draft row, logits row) when given."""
    V = vocab if vocab is not None else w.V
    Lm, Lb = w.L_max, w.L[b]
    draft, logits = out if out is not None else (torch.zeros((Lm,), dtype=torch.int32, device=device),
                                                 torch.empty((Lm + 1, V), dtype=torch.float32, device=device))
    gd = _gen(w, rnd, b, KIND_DRAFT, device)
    draft[:Lb] = torch.randint(0, V, (Lb,), generator=gd, device=device, dtype=torch.int64).to(torch.int32)
    gl = _gen(w, rnd, b, KIND_LOGITS, device)
    logits[:] = torch.randn((Lm + 1, V), generator=gl, device=device, dtype=torch.float32)
    gp = _gen(w, rnd, b, KIND_PLANT, device)
    u = torch.rand((Lm,), generator=gp, device=device, dtype=torch.float64)
    rows = logits[:Lb]
    x = draft[:Lb].long()
    rmax = rows.max(dim=1).values
    rmin = rows.min(dim=1).values
    am = rows.argmax(dim=1)
    plant = u[:Lb] < w.p[b]
    ar = torch.arange(Lb, device=device)
    hit = torch.where(plant, rmax + 1.0, torch.where(am == x, rmin - 1.0, rows[ar, x]))
    rows[ar, x] = hit
    return draft, logits


def drafts_and_logits(w: Workload, rnd: int, device="cpu", vocab: int | None = None):
    """(draft int32 [B][L_max], logits fp32 [B][L_max+1][V], L int32 [B]) with planted matches."""
    V = vocab if vocab is not None else w.V
    B, Lm = w.B, w.L_max
    draft = torch.zeros((B, Lm), dtype=torch.int32, device=device)
    logits = torch.empty((B, Lm + 1, V), dtype=torch.float32, device=device)
    for b in range(B):
        request_logits(w, rnd, b, device, V, out=(draft[b], logits[b]))
    Lt = torch.tensor(w.L, dtype=torch.int32, device=device)
    return draft, logits, Lt
