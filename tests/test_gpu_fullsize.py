"""Full-size parity for the two largest workloads, against the float64 oracle on sampled heads.

Llama-70B long-context offload (4 requests x 131,072 tokens, 64/8 heads, 4-bit KV_comp, L 40): the
4-bit draft on sampled (step, KV head) and the verification of 320 query rows per KV head (three
128-row tiles) at full context.

Mixed staggered serving batch (32 requests, contexts 8K-256K, half token drop 4x and half 2-bit,
KV_full of half of them staged from pinned host memory, L 25-40): run whole through the engine's
two-group stagger -- one draft call per compression mode and step, the host-resident caches copied
over the host link every period -- for 20 rounds with per-round inputs. Accept is compared bit for
bit on every request of every round; draft and verify attention on rounds 0 and 19 for sampled
requests and KV heads ("VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core
algorithm", "Architecture support", "Cross-resource staggering (P1)").
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from workloads import configs, gen, DROP
from tests.util import make_batch, f32, assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _oracle_head(w, b, r, hk):
    """The oracle's KV_comp main rows and initial window of request b on KV head hk only (float32)."""
    kf, vf = f32(r.k_full[hk:hk + 1, : w.ctx[b]]), f32(r.v_full[hk:hk + 1, : w.ctx[b]])
    if w.mode[b] == DROP:
        idx = O.keep_set(r.importance.cpu().numpy()[: w.ctx[b]], w.keep[b], w.recent[b])
        km, vm = O.comp_main_rows("drop", kf, vf, idx=idx)
        z = np.zeros((1, 0, w.d), np.float32)
        return kf, vf, km, vm, z, z
    qkv = O.quantize_kv(kf, vf, w.bits, w.residual_min)
    km, vm = O.comp_main_rows("quant", kf, vf, qkv=qkv)
    return kf, vf, km, vm, qkv["k_res"], qkv["v_res"]


def _check_draft(w, b, r, hk, steps, what, q=None, kn=None, vn=None, heads=None):
    G = w.Hq // w.Hkv
    kf, vf, km, vm, kw0, vw0 = heads[hk] if heads is not None else _oracle_head(w, b, r, hk)
    q = f32(r.q) if q is None else q
    kn = f32(r.k_new) if kn is None else kn
    vn = f32(r.v_new) if vn is None else vn
    sel = slice(hk * G, (hk + 1) * G)
    for s in steps:
        kw = np.concatenate([kw0, kn[: s + 1, hk:hk + 1].transpose(1, 0, 2)], axis=1)
        vw = np.concatenate([vw0, vn[: s + 1, hk:hk + 1].transpose(1, 0, 2)], axis=1)
        ref = O.draft_attn(q[s, sel], km, vm, kw, vw)
        assert_attn_close(r.o_draft[s, sel], ref, f"{what} draft b{b} s{s} hk{hk}")


def _check_verify(w, b, r, hk, what, q=None, kn=None, vn=None, heads=None):
    G = w.Hq // w.Hkv
    kf, vf = heads[hk][:2] if heads is not None else (f32(r.k_full[hk:hk + 1, : w.ctx[b]]),
                                                      f32(r.v_full[hk:hk + 1, : w.ctx[b]]))
    q = f32(r.q) if q is None else q
    kn = f32(r.k_new) if kn is None else kn
    vn = f32(r.v_new) if vn is None else vn
    sel = slice(hk * G, (hk + 1) * G)
    ref = O.verify_attn(q[:, sel], kf, vf, kn[:, hk:hk + 1].transpose(1, 0, 2), vn[:, hk:hk + 1].transpose(1, 0, 2))
    assert_attn_close(r.o_verify[:, sel], ref, f"{what} verify b{b} hk{hk}")


def test_llama70b_offload_full_size_sampled():
    """4 x 131,072 tokens, 4-bit (4,092 blocks per head): all 40 draft steps run, steps 0 and 39
    checked on two KV heads; then the verification (3 row tiles of 128 rows per KV head) checked
    on one KV head of every request, and again in trio mode (VC_VERIFY_TRIO=1: every K/V tile read
    once for the three row tiles) on two requests."""
    w = configs.llama70b_offload4()
    bt = make_batch(w, list(range(w.B)))
    bt.compress()
    for s in range(w.L_max):
        bt.draft_step(s)
    bt.verify()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    for b in range(w.B):
        r = bt.reqs[b]
        if b in (0, 3):
            for hk in (0, 7) if b == 0 else (5,):
                _check_draft(w, b, r, hk, [0, w.L[b] - 1], w.name)
        _check_verify(w, b, r, (2 * b + 1) % w.Hkv, w.name)
    # the same verification with every K/V tile read once for the three row tiles (trio mode)
    os.environ["VC_VERIFY_TRIO"] = "1"
    try:
        for r in bt.reqs:
            r.o_verify.zero_()
        bt.verify()
        torch.cuda.synchronize()
    finally:
        del os.environ["VC_VERIFY_TRIO"]
    assert int(bt.dev_status.item()) == 0
    for b in (1, 2):
        _check_verify(w, b, bt.reqs[b], (2 * b + 1) % w.Hkv, w.name + " trio")


def test_mixed_serving_whole_twenty_rounds():
    from lossless_compressed_kv_vc_gb300 import engine, VC_TOKEN_DROP, VC_QUANT
    w = configs.mixed_serving()
    dev = "cuda"
    reqs = []
    for b in range(w.B):
        ri = gen.request(w, 0, b, dev)
        drop = w.mode[b] == DROP
        reqs.append(engine.Req(mode=VC_TOKEN_DROP if drop else VC_QUANT, ctx=w.ctx[b], L=w.L[b], k_full=ri.k_full,
                               v_full=ri.v_full, q=ri.q, k_new=ri.k_new, v_new=ri.v_new,
                               importance=ri.importance if drop else None, keep=w.keep[b], recent=w.recent[b],
                               compact=bool(drop and w.on_host[b]), bits=w.bits))
    del ri
    # the oracle's KV_comp of the sampled requests and heads, while KV_full is still in HBM
    samples = {}
    for m in (DROP, "quant"):
        for host in (False, True):
            b = next(b for b in range(w.B) if w.mode[b] == m and w.on_host[b] == host)
            hk = b % w.Hkv
            samples[b] = (hk, {hk: _oracle_head(w, b, reqs[b], hk)})
    # the planner's split, on costs proportional to each request's bytes (draft, verify, copy)
    d = w.d
    cost = lambda b: (w.L[b] * (w.ctx[b] // 4 * 4096 if w.mode[b] == DROP else w.ctx[b] * 768),
                      w.ctx[b] * 4096, w.ctx[b] * 4096 * 30 if w.on_host[b] else 0)
    g0, g1, _ = engine.plan_groups(engine.stagger_costs(*zip(*[cost(b) for b in range(w.B)])))
    split = [0 if b in g0 else 1 for b in range(w.B)]
    assert g0 and g1
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    groups, members, host_kv, slots = engine.staggered_groups(w.Hq, w.Hkv, d, reqs, split, w.on_host,
                                                              w.residual_min, dev, ks)
    assert sum(h is not None for g in host_kv for h in g) == sum(w.on_host)
    draft, logits, Lt = gen.drafts_and_logits(w, 0, dev)
    io = engine.group_io(members, logits, draft, Lt)
    sg = engine.StaggeredOffload(groups, host_kv, slots, cs, ks)
    rounds = 20

    def load(gi, rnd):
        """Round rnd's inputs of group gi into its tensors, in order on the compute stream."""
        with torch.cuda.stream(ks):
            for j, idx in enumerate(members[gi]):
                bt = groups[gi][j]
                lg, dr, L, _, _ = io[gi][j]
                for i, b in enumerate(idx):
                    q, kn, vn = gen.round_queries(w, rnd, b, dev)
                    r = bt.reqs[i]
                    r.q.copy_(q)
                    r.k_new.copy_(kn)
                    r.v_new.copy_(vn)
                    gen.request_logits(w, rnd, b, dev, out=(dr[i], lg[i]))

    def check(gi, rnd):
        """Group gi's round rnd has been drafted, verified and accepted."""
        torch.cuda.synchronize()
        for bt in groups[gi]:
            assert int(bt.dev_status.item()) == 0
        for j, idx in enumerate(members[gi]):
            lg, dr, L, tok, nacc = io[gi][j]
            lg_np, dr_np, tok_np, nacc_np = lg.cpu().numpy(), dr.cpu().numpy(), tok.cpu().numpy(), nacc.cpu().numpy()
            for i, b in enumerate(idx):
                ref_tok, ref_n = O.accept(lg_np[i], dr_np[i], w.L[b])
                assert int(nacc_np[i]) == ref_n, (rnd, b)
                assert tok_np[i, :ref_n].tolist() == ref_tok and (tok_np[i, ref_n:] == -1).all(), (rnd, b)
                if rnd in (0, rounds - 1) and b in samples:
                    hk, heads = samples[b]
                    r = groups[gi][j].reqs[i]  # its q, k_new, v_new still hold round rnd's inputs
                    _check_draft(w, b, r, hk, [0, w.L[b] // 2, w.L[b] - 1], f"round {rnd}", heads=heads)
                    _check_verify(w, b, r, hk, f"round {rnd}", heads=heads)

    # group 0 drafts round r in phase 0 and is verified in phase 1 of the same period; group 1
    # drafts round r in phase 1 and is verified in phase 0 of the next period
    for rnd in range(rounds + 1):
        if rnd < rounds:
            load(0, rnd)
        sg.phase(0, io)
        if rnd > 0:
            check(1, rnd - 1)
        if rnd == rounds:
            break
        load(1, rnd)
        sg.phase(1, io)
        check(0, rnd)
