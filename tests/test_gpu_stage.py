"""Staging KV_full from pinned host memory (vc_stage_full_kv) and the staggered offload round:
one group drafts while the other group's KV_full crosses the host link, then is verified
("VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Cross-resource staggering (P1)",
"Architecture support": long-context decoding with KV_full in CPU memory)."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import configs, gen
from tests.util import make_batch, f32, assert_attn_close, oracle_main

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__ as g
    g.build()
    import lossless_compressed_kv_vc_gb300 as m
    return m


@pytest.mark.parametrize("nbytes,chunk", [(37 * (1 << 20) + 48, 1 << 20), (4096, 0), (3 << 20, 5 << 20)])
def test_stage_copies_every_byte(vc, nbytes, chunk):
    host = torch.randint(0, 256, (nbytes,), dtype=torch.uint8).pin_memory()
    dev = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    cs = torch.cuda.Stream()
    done = torch.cuda.Event()
    vc.vc_stage_full_kv(host, dev, nbytes, chunk, cs, done)
    torch.cuda.current_stream().wait_event(done)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)


def test_stage_refuses_pageable_source(vc):
    """A host buffer that is not page-locked is refused before any copy is issued."""
    host = torch.ones(1 << 16, dtype=torch.uint8)  # pageable
    dev = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    st = vc.vc_stage_full_kv(host, dev, host.numel(), 0, torch.cuda.current_stream(), None, raise_on_error=False)
    assert st == vc.VC_ERR_NOT_PINNED
    torch.cuda.synchronize()
    assert int(dev.sum()) == 0


def test_stage_refuses_device_source(vc):
    a = torch.ones(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert vc.vc_stage_full_kv(a, b, 4096, 0, None, None, raise_on_error=False) == vc.VC_ERR_NOT_PINNED


@pytest.mark.parametrize("head_chunks,graphs", [(1, False), (3, False), (8, False), (1, True)])
def test_staggered_offload_period_matches_oracle(vc, head_chunks, graphs):
    """Scaled Llama-70B-shape offload workload (4 requests, 64/8 heads, 4-bit): a full period of the
    two-group stagger gives the oracle's draft outputs, verify outputs and accepted tokens, with
    the copy staged whole (1) or a KV-head range at a time and verified range by range (3: uneven
    ranges of 2, 3 and 3 heads; 8: one head per range), and with each group's draft series
    replayed from a captured CUDA graph."""
    from lossless_compressed_kv_vc_gb300 import engine
    w = configs.scaled(configs.llama70b_offload4(), ctx_div=64, batch=4, L=6)
    w.V = 5000
    groups = [make_batch(w, [0, 1]), make_batch(w, [2, 3])]
    full_ref = {}
    for gi, bt in enumerate(groups):
        for i, r in enumerate(bt.reqs):
            full_ref[2 * gi + i] = (f32(r.k_full), f32(r.v_full))
        bt.compress()
    host_kv, slots = engine.move_full_kv_to_host(groups)
    for bt in groups:
        bt.prepare_steps()
    draft, logits, L = gen.drafts_and_logits(w, 0, "cuda")
    io = []
    for gi in range(2):
        sl = slice(2 * gi, 2 * gi + 2)
        io.append((logits[sl].contiguous(), draft[sl].contiguous(), L[sl].contiguous(),
                   torch.empty((2, w.L_max + 1), dtype=torch.int32, device="cuda"),
                   torch.empty((2,), dtype=torch.int32, device="cuda")))
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    # the period verifies what each group drafted in the previous phase: draft group 1 first
    for shape, arr, act in groups[1]._steps:
        vc.vc_draft_attn(shape, arr, groups[1].ws_draft, groups[1].dev_status, ks)
    ks.synchronize()
    sg = engine.StaggeredOffload(groups, host_kv, slots, cs, ks, chunk_bytes=1 << 20, head_chunks=head_chunks)
    if graphs:  # each group's draft series replayed as a captured CUDA graph
        sg.capture_drafts()
        assert len(sg._graphs) == 2
    sg.period(io)
    torch.cuda.synchronize()
    for gi, bt in enumerate(groups):
        assert int(bt.dev_status.item()) == 0
        for i, r in enumerate(bt.reqs):
            b = 2 * gi + i
            kf, vf = full_ref[b]
            assert torch.equal(slots[gi][i].cpu(), host_kv[gi][i])  # staged bytes
            km, vm, kw0, vw0 = oracle_main(w, b, kf, vf)
            ref_d = O.draft_round(f32(r.q), km, vm, kw0, vw0, f32(r.k_new), f32(r.v_new))
            assert_attn_close(r.o_draft, ref_d, f"draft b{b}")
            ref_v = O.verify_attn(f32(r.q), kf, vf, f32(r.k_new).transpose(1, 0, 2), f32(r.v_new).transpose(1, 0, 2))
            assert_attn_close(r.o_verify, ref_v, f"verify b{b}")
        lg, dr, Lg, tok, nacc = io[gi]
        for i in range(2):
            rt, rn = O.accept(lg[i].cpu().numpy(), dr[i].cpu().numpy(), int(Lg[i]))
            assert int(nacc[i]) == rn and tok[i, :rn].cpu().tolist() == rt


def test_round_from_host_matches_device_round_and_oracle(vc):
    """The engine's host-input round (inputs copied from pinned host memory, the accept inputs on a
    second stream under the draft phase) gives bit-identical draft and verify outputs to the
    device-resident round, and the oracle's accepted tokens in two successive rounds whose host
    logits differ; a third round reuses the first round's device slot, whose copies must wait
    for that round's accept."""
    from lossless_compressed_kv_vc_gb300 import engine
    w = configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=3, L=8)
    w.V = 5000
    bt = make_batch(w, [0, 1, 2])
    bt.compress()
    bt.prepare_steps()
    draft, logits, L = gen.drafts_and_logits(w, 0, device="cuda")
    tok = torch.empty((w.B, w.L_max + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((w.B,), dtype=torch.int32, device="cuda")
    bt.run_round(logits, draft, L, tok, nacc, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref_d = [r.o_draft.clone() for r in bt.reqs]
    ref_v = [r.o_verify.clone() for r in bt.reqs]
    hr = engine.HostRound(bt, logits, draft, L, tok, nacc)
    for r in bt.reqs:  # the round must use what it copies
        for t in (r.q, r.k_new, r.v_new, r.importance, r.o_draft, r.o_verify):
            t.zero_()
    for t in (draft, logits, L, tok, nacc):
        t.zero_()
    cs = torch.cuda.Stream()
    s = torch.cuda.current_stream()
    for rnd in (0, 1, 2):
        d_h, l_h, L_h = gen.drafts_and_logits(w, rnd)
        for (h, _), src in zip(hr.accept_inputs, (d_h, l_h, L_h)):
            h.copy_(src)
        bt.run_round_from_host(hr, s, cs)
        torch.cuda.synchronize()
        assert int(bt.dev_status.item()) == 0
        if rnd == 0:
            for b in range(w.B):
                assert torch.equal(bt.reqs[b].o_draft, ref_d[b])
                assert torch.equal(bt.reqs[b].o_verify, ref_v[b])
        lg, dr = l_h.numpy(), d_h.numpy()
        for b in range(w.B):
            rt, rn = O.accept(lg[b], dr[b], w.L[b])
            assert int(hr.host_n_acc[b]) == rn, (rnd, b)
            assert hr.host_tokens[b, :rn].tolist() == rt


def test_planned_stagger_with_resident_requests_matches_oracle(vc):
    """Six 2-bit requests of the mixed serving workload (scaled), three with KV_full on the host and
    three resident: groups from the planner, one period; drafts, verifications and accepted tokens
    match the oracle, and the host requests' slots hold the staged bytes."""
    from lossless_compressed_kv_vc_gb300 import engine
    full = configs.mixed_serving()
    w = configs.subset(full, full.request_indices("quant")[:6])
    w = configs.scaled(w, ctx_div=64, L=5)
    w.V = 3000
    reqs, host, slot, ref = [], [], [], []
    for b in range(w.B):
        ri = gen.request(w, 0, b, "cuda")
        ref.append((f32(ri.k_full), f32(ri.v_full)))
        kf, vf, h, s = ri.k_full, ri.v_full, None, None
        if w.on_host[b]:
            s = torch.stack([kf, vf])
            h = torch.empty(s.shape, dtype=s.dtype, pin_memory=True)
            h.copy_(s)
            kf, vf = s[0], s[1]
        host.append(h)
        slot.append(s)
        reqs.append(engine.Req(mode=vc.VC_QUANT, ctx=w.ctx[b], L=w.L[b], k_full=kf, v_full=vf, q=ri.q,
                               k_new=ri.k_new, v_new=ri.v_new, bits=w.bits))
    costs = engine.stagger_costs([w.ctx[b] * w.L[b] for b in range(w.B)], [w.ctx[b] for b in range(w.B)],
                                 [8 * w.ctx[b] if w.on_host[b] else 0 for b in range(w.B)])
    g0, g1, _ = engine.plan_groups(costs)
    assert g0 and g1
    idx = [g0, g1]
    groups = [engine.Batch(w.Hq, w.Hkv, w.d, [reqs[b] for b in ix], residual_min=w.residual_min) for ix in idx]
    for bt in groups:
        bt.compress()
        bt.prepare_steps()
    draft, logits, L = gen.drafts_and_logits(w, 0, "cuda")
    io = []
    for ix in idx:
        sel = torch.tensor(ix, device="cuda")
        io.append((logits[sel].contiguous(), draft[sel].contiguous(), L[sel].contiguous(),
                   torch.empty((len(ix), w.L_max + 1), dtype=torch.int32, device="cuda"),
                   torch.empty((len(ix),), dtype=torch.int32, device="cuda")))
    for s in slot:  # the staged copies must bring the bytes back
        if s is not None:
            s.zero_()
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    for shape, arr, act in groups[1]._steps:
        vc.vc_draft_attn(shape, arr, groups[1].ws_draft, groups[1].dev_status, ks)
    ks.synchronize()
    sg = engine.StaggeredOffload(groups, [[host[b] for b in ix] for ix in idx], [[slot[b] for b in ix] for ix in idx],
                                 cs, ks, chunk_bytes=1 << 20)
    sg.period(io)
    torch.cuda.synchronize()
    for gi, (bt, ix) in enumerate(zip(groups, idx)):
        assert int(bt.dev_status.item()) == 0
        lg, dr, Lg, tok, nacc = io[gi]
        for i, b in enumerate(ix):
            r = bt.reqs[i]
            kf, vf = ref[b]
            if host[b] is not None:
                assert torch.equal(slot[b].cpu(), host[b])
            km, vm, kw0, vw0 = oracle_main(w, b, kf, vf)
            assert_attn_close(r.o_draft, O.draft_round(f32(r.q), km, vm, kw0, vw0, f32(r.k_new), f32(r.v_new)),
                              f"draft b{b}")
            ref_v = O.verify_attn(f32(r.q), kf, vf, f32(r.k_new).transpose(1, 0, 2), f32(r.v_new).transpose(1, 0, 2))
            assert_attn_close(r.o_verify, ref_v, f"verify b{b}")
            rt, rn = O.accept(lg[i].cpu().numpy(), dr[i].cpu().numpy(), int(Lg[i]))
            assert int(nacc[i]) == rn and tok[i, :rn].cpu().tolist() == rt


def test_batch_calls_on_another_stream_follow_its_construction(vc):
    """A Batch is built on the current stream (KV_full written, windows and workspace zero-filled
    there) and then compressed and drafted on a side stream, as the staggered round does. The side
    stream must start after that work: here the current stream is held back by a bounded sleep
    kernel before the inputs are even generated, so without the ordering the compress would read
    KV_full before it is written or have its residual window wiped by a late zero fill. Codes,
    scales, zeros and the window are compared bit for bit with the oracle's quantisation, and the
    first draft step with the oracle's attention."""
    from tests.util import assert_quant_state
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=64, batch=2, L=2)
    ks = torch.cuda.Stream()
    torch.cuda._sleep(100_000_000)  # about 50 ms of device time on the current stream
    bt = make_batch(w, list(range(w.B)))
    bt.compress(ks)
    bt.draft_step(0, ks)
    ks.synchronize()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    bt.reset_window()  # the window counts as after compress (the draft step appended a row)
    for i in range(w.B):
        r = bt.reqs[i]
        kf, vf = f32(r.k_full[:, : w.ctx[i]]), f32(r.v_full[:, : w.ctx[i]])
        assert_quant_state(bt, i, kf, vf, w.bits, w.residual_min)
        km, vm, kw0, vw0 = oracle_main(w, i, kf, vf)
        kn, vn = f32(r.k_new[:1]).transpose(1, 0, 2), f32(r.v_new[:1]).transpose(1, 0, 2)
        ref = O.draft_attn(f32(r.q[0]), km, vm, np.concatenate([kw0, kn], 1), np.concatenate([vw0, vn], 1))
        assert_attn_close(r.o_draft[0], ref, f"request {i} on a side stream")
