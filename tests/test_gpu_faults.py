"""Failure detection without a GPU fault: a staging copy that fails on the host side, and a draft
wait that runs out on the device.

Staging ("Architecture support": KV_full crosses the host link for verification): the test hook
VC_FAIL_STAGE_CHUNK makes vc_stage_full_kv treat one chunk's cudaMemcpyAsync as failed; the call
returns VC_ERR_CUDA, the chunks before it land, nothing after it is issued, and the next call
without the hook copies everything.

Draft (the kernel's bounded waits): VC_SPIN_LIMIT=0 makes every warp's wait for its first stage
of data give up at once. Each warp records VC_DEV_TIMEOUT, still waits for the copies it issued
(so none is in flight when its CTA exits), skips its range, and the launch completes with finite
outputs. The same process then runs the step again without the limit and matches the oracle:
the context stays usable. Nothing here traps, faults or hangs.
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import configs
from tests.util import make_batch, f32, assert_attn_close, oracle_main

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__ as g
    g.build()
    import lossless_compressed_kv_vc_gb300 as m
    return m


def test_stage_reports_a_failed_chunk_and_issues_nothing_after_it(vc, monkeypatch):
    mb = 1 << 20
    host = torch.randint(0, 256, (5 * mb + 100,), dtype=torch.uint8).pin_memory()
    dev = torch.zeros(host.numel(), dtype=torch.uint8, device="cuda")
    cs = torch.cuda.Stream()
    monkeypatch.setenv("VC_FAIL_STAGE_CHUNK", "2")
    st = vc.vc_stage_full_kv(host, dev, host.numel(), mb, cs, None, raise_on_error=False)
    assert st == vc.VC_ERR_CUDA
    cs.synchronize()
    got = dev.cpu()
    assert torch.equal(got[: 2 * mb], host[: 2 * mb])      # chunks 0 and 1 were issued
    assert int(got[2 * mb:].count_nonzero()) == 0          # chunk 2 failed, nothing after it issued
    monkeypatch.delenv("VC_FAIL_STAGE_CHUNK")
    done = torch.cuda.Event()
    assert vc.vc_stage_full_kv(host, dev, host.numel(), mb, cs, done) == vc.VC_OK
    done.synchronize()
    assert torch.equal(dev.cpu(), host)


@pytest.mark.parametrize("which", ["drop", "quant", "quant_tc"])
def test_draft_wait_runs_out_then_the_context_stays_usable(vc, monkeypatch, which):
    """quant_tc: the tcgen05 draft kernel (VC_DRAFT_TC=1), whose roles give up together through a
    shared flag, wait for their copies and MMAs, free TMEM and leave zero (finite) outputs."""
    monkeypatch.setenv("VC_DRAFT_TC", "1" if which == "quant_tc" else "0")
    if which == "drop":
        w = configs.scaled(configs.llama8b_drop(), ctx_div=32, batch=2, L=2)
    else:
        w = configs.scaled(configs.qwen32b_quant2(), ctx_div=64, batch=2, L=2)
    bt = make_batch(w, list(range(w.B)))
    bt.compress()
    torch.cuda.synchronize()
    monkeypatch.setenv("VC_SPIN_LIMIT", "0")
    bt.draft_step(0)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == vc.VC_DEV_TIMEOUT
    for r in bt.reqs:
        assert torch.isfinite(r.o_draft[0].float()).all()
    # the same step again, no limit: the oracle's output
    monkeypatch.delenv("VC_SPIN_LIMIT")
    bt.dev_status.zero_()
    bt.reset_window()
    bt.draft_step(0)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    for i, b in enumerate(range(w.B)):
        r = bt.reqs[i]
        imp = None if r.importance is None else r.importance.cpu().numpy()
        km, vm, kw0, vw0 = oracle_main(w, b, f32(r.k_full), f32(r.v_full), imp)
        kn, vn = f32(r.k_new[:1]).transpose(1, 0, 2), f32(r.v_new[:1]).transpose(1, 0, 2)
        ref = O.draft_attn(f32(r.q[0]), km, vm, np.concatenate([kw0, kn], 1), np.concatenate([vw0, vn], 1))
        assert_attn_close(r.o_draft[0], ref, f"{which} request {b} after a timed-out launch")
