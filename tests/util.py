"""Test plumbing: building requests from the seeded workloads, and the float tolerance.

Tolerance for attention outputs (bf16 I/O, fp32 accumulation): each element must satisfy
|gpu - oracle| <= max(1e-2, 2e-2 * |oracle|) (max-abs 1e-2 or max-rel 2e-2), oracle in float64.
Integer, index and byte outputs are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from workloads import gen, DROP, QUANT

ATOL, RTOL = 1e-2, 2e-2


def assert_attn_close(gpu, ref, what=""):
    g = gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    lim = np.maximum(ATOL, RTOL * np.abs(r))
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu {g[i]:.6g} oracle {r[i]:.6g} (max abs err {err.max():.3g})")
    return float(err.max())


def make_batch(w, reqs, rnd=0, device="cuda", compact=False):
    """Engine Batch for requests `reqs` of workload w, inputs from the seeded generator."""
    from lossless_compressed_kv_vc_gb300 import engine, VC_TOKEN_DROP, VC_QUANT
    rs = []
    for b in reqs:
        ri = gen.request(w, rnd, b, device)
        mode = VC_TOKEN_DROP if w.mode[b] == DROP else VC_QUANT
        rs.append(engine.Req(mode=mode, ctx=w.ctx[b], L=w.L[b], k_full=ri.k_full, v_full=ri.v_full, q=ri.q,
                             k_new=ri.k_new, v_new=ri.v_new, importance=ri.importance, keep=w.keep[b],
                             recent=w.recent[b], compact=compact, bits=w.bits))
    return engine.Batch(w.Hq, w.Hkv, w.d, rs, residual_min=w.residual_min, device=device)


def f32(t):
    return t.detach().to("cpu").to(torch.float32).numpy()


def oracle_main(w, b, k_full_f32, v_full_f32, importance=None):
    """The oracle's KV_comp main rows and initial window for request b of workload w."""
    import oracle as O
    if w.mode[b] == DROP:
        idx = O.keep_set(importance, w.keep[b], w.recent[b])
        km, vm = O.comp_main_rows("drop", k_full_f32, v_full_f32, idx=idx)
        z = np.zeros((w.Hkv, 0, w.d), np.float32)
        return km, vm, z, z
    qkv = O.quantize_kv(k_full_f32, v_full_f32, w.bits, w.residual_min)
    km, vm = O.comp_main_rows("quant", k_full_f32, v_full_f32, qkv=qkv)
    return km, vm, qkv["k_res"], qkv["v_res"]
