"""Test plumbing: building requests from the seeded workloads, and the float tolerance.

Tolerance for attention outputs (bf16 I/O, fp32 accumulation), oracle in float64. Three checks:
  1. every element: |gpu - oracle| <= max(1e-2, 2e-2 * |oracle|) (max-abs 1e-2 or max-rel 2e-2);
  2. every head (the outputs of one query head, over all rows compared): relative L2 error
     ||gpu - oracle|| / ||oracle|| <= 5e-3;
  3. every element: |gpu - oracle| <= 2^-6 |oracle| + 2^-6 rms(oracle's output vector holding it),
     the vector being one query row's d outputs for one head (each has its own scale: a row that
     one key dominates is as large as that key's value row).
Check 1 alone cannot see a kernel that loses a few chunks of a long keep-set: at 8192 kept rows the
outputs have a standard deviation near 0.011, far below its 1e-2 floor, while dropping 64 of the
rows or scaling the scores by 0.95 moves them by several percent (tests/test_tolerance.py plants
both mistakes and checks that they fail here). A correct kernel rounds twice: the attention weights
P to bf16 (fp16 in the quantised draft) as the operand of the P V product, and the output to bf16,
each after fp32 accumulation. Check 3 allows 2^-7 for each rounding: on the CPU, that arithmetic
(bf16 P, fp32 sums, bf16 output) reaches 0.9 of a single 2^-7 over 790K elements of the four
verify row tile case, and one GPU element of 1.6M reached 1.02 of it.
Integer, index and byte outputs are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from workloads import gen, DROP, QUANT

ATOL, RTOL = 1e-2, 2e-2
REL_L2 = 5e-3
TIGHT = 2.0 ** -6


def _by_head(a):
    """[heads][rest] view: the second-to-last axis holds the query heads ([rows][heads][d] or
    [heads][d]); a 1-D array is one head."""
    if a.ndim == 1:
        return a[None, :]
    return np.moveaxis(a, -2, 0).reshape(a.shape[-2], -1)


def attn_errors(gpu, ref):
    """Each check's violations: (elements out of check 1, worst per-head relative L2 error,
    elements out of check 3, and a description of check 3's worst element)."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    n1 = int((err > np.maximum(ATOL, RTOL * np.abs(r))).sum())
    gh, rh = _by_head(g), _by_head(r)
    eh = np.abs(gh - rh)
    nrm = np.sqrt((rh * rh).sum(axis=1))
    rel = np.sqrt((eh * eh).sum(axis=1)) / np.maximum(nrm, 1e-30)
    rms = np.sqrt((r * r).mean(axis=-1, keepdims=True))  # per output vector (last axis = d)
    lim3 = TIGHT * np.abs(r) + TIGHT * rms
    n3 = int((err > lim3).sum())
    i = np.unravel_index(np.argmax(err / np.maximum(lim3, 1e-300)), err.shape)
    worst = f"worst at {i}: gpu {g[i]:.6g} oracle {r[i]:.6g} err {err[i]:.3g} bound {lim3[i]:.3g}"
    return n1, float(rel.max()), n3, worst


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
    _, rel, n3, worst = attn_errors(g, r)
    if rel > REL_L2:
        raise AssertionError(f"{what}: relative L2 error {rel:.3g} of a head exceeds {REL_L2}")
    if n3:
        raise AssertionError(f"{what}: {n3} elements beyond 2^-6 |oracle| + 2^-6 rms(oracle's output vector); {worst}")
    return float(err.max())


def make_batch(w, reqs, rnd=0, device="cuda", compact=False, grow=0):
    """Engine Batch for requests `reqs` of workload w, inputs from the seeded generator. With
    grow > 0 each KV_full (and importance array) has room for `grow` more tokens."""
    from lossless_compressed_kv_vc_gb300 import engine, VC_TOKEN_DROP, VC_QUANT
    rs = []
    for b in reqs:
        ri = gen.request(w, rnd, b, device)
        kf, vf, imp = ri.k_full, ri.v_full, ri.importance
        if grow > 0:
            kf = torch.zeros((w.Hkv, w.ctx[b] + grow, w.d), dtype=torch.bfloat16, device=device)
            vf = torch.zeros_like(kf)
            kf[:, : w.ctx[b]] = ri.k_full
            vf[:, : w.ctx[b]] = ri.v_full
            if imp is not None:
                imp = gen.importance(w, b, device, n=w.ctx[b] + grow)
        mode = VC_TOKEN_DROP if w.mode[b] == DROP else VC_QUANT
        rs.append(engine.Req(mode=mode, ctx=w.ctx[b], L=w.L[b], k_full=kf, v_full=vf, q=ri.q,
                             k_new=ri.k_new, v_new=ri.v_new, importance=imp, keep=w.keep[b],
                             recent=w.recent[b], compact=compact, bits=w.bits, grow=grow))
    return engine.Batch(w.Hq, w.Hkv, w.d, rs, residual_min=w.residual_min, device=device)


def f32(t):
    return t.detach().to("cpu").to(torch.float32).numpy()


def assert_quant_state(bt, i, kf, vf, bits, residual_min):
    """Request i of Batch bt holds, bit for bit, the oracle's quantisation of the float32 cache
    kf, vf [Hkv][ctx][d]: block count, codes, fp16 scales and zeros, and the residual window."""
    import oracle as O
    r, c = bt.reqs[i], bt.comp[i]
    ref = O.quantize_kv(kf, vf, bits, residual_min)
    ng = ref["ng"]
    assert (c.ng, c.n_win) == (ng, ref["n_res"]), (c.ng, c.n_win, ng, ref["n_res"])
    if ng > 0:
        u16 = lambda t: t.cpu().numpy().view(np.uint16)
        assert np.array_equal(r.kc[:, :ng].cpu().numpy(), ref["kc"])
        assert np.array_equal(u16(r.ks[:, :ng]), ref["ks"].view(np.uint16))
        assert np.array_equal(u16(r.kz[:, :ng]), ref["kz"].view(np.uint16))
        assert np.array_equal(r.vc[:, :ng].cpu().numpy(), ref["vc"])
        assert np.array_equal(u16(r.vs[:, : 32 * ng]), ref["vs"].view(np.uint16))
        assert np.array_equal(u16(r.vz[:, : 32 * ng]), ref["vz"].view(np.uint16))
    assert np.array_equal(f32(r.k_win[:, : ref["n_res"]]), ref["k_res"])
    assert np.array_equal(f32(r.v_win[:, : ref["n_res"]]), ref["v_res"])
    return ref


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
