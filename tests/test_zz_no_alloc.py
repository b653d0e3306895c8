"""vc_draft_attn_noalloc: the draft step for callers that cannot allocate device memory (a plugin
whose host application owns all device allocations, or a loop that must not call cudaMalloc).

It is called through the C ABI and must give the same output as vc_draft_attn with a caller
workspace, within the attention tolerance the other tests use, and match the oracle, on calls in a
row. The shared scratch array keeps each call's data for the next one, so the calls change shape
between them: the number of KV heads grows (2 -> 8), shrinks and grows again, which moves where a
shape-dependent layout would put the partials. This file sorts last so a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from workloads import configs
from tests.util import make_batch, assert_attn_close, f32, oracle_main

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__ as g
    g.build()
    import lossless_compressed_kv_vc_gb300 as m
    return m


def _case(name):
    if name == "tiny":  # Hkv 2, d 64
        return configs.scaled(configs.tiny(), batch=1, L=2)
    if name == "drop8":  # Hkv 8, d 128, token drop
        return configs.scaled(configs.llama8b_drop(), ctx_div=8, batch=4, L=2)
    return configs.scaled(configs.qwen32b_quant2(), ctx_div=16, batch=3, L=2)  # Hkv 8, G 5, 2-bit


def _noalloc(vc, shape, arr, status):
    lib = vc.lib_handle()
    return lib.vc_draft_attn_noalloc(ctypes.byref(shape), arr, ctypes.c_void_p(status.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_steps(vc, name):
    """Two draft steps of one batch: each through the workspace entry point, then through the
    no-allocation one (outputs cleared in between), compared with each other and with the oracle."""
    w = _case(name)
    bt = make_batch(w, list(range(w.B)))
    bt.compress()
    torch.cuda.synchronize()
    mains = [oracle_main(w, b, f32(bt.reqs[b].k_full[:, : w.ctx[b]]), f32(bt.reqs[b].v_full[:, : w.ctx[b]]),
                         None if bt.reqs[b].importance is None else bt.reqs[b].importance.cpu().numpy())
             for b in range(w.B)]
    for step in range(2):
        act, arr = bt.draft_requests(step)
        shape = vc.vc_shape(len(act), w.Hq, w.Hkv, w.d)
        vc.vc_draft_attn(shape, arr, bt.ws_draft, bt.dev_status)
        torch.cuda.synchronize()
        ref = [bt.reqs[b].o_draft[step].clone() for b in act]
        for b in act:
            bt.reqs[b].o_draft[step].fill_(float("nan"))
        st = _noalloc(vc, shape, arr, bt.dev_status)
        assert st == vc.VC_OK, vc.vc_status_string(st)
        torch.cuda.synchronize()
        assert int(bt.dev_status.item()) == 0
        for i, b in enumerate(act):
            r = bt.reqs[b]
            assert_attn_close(r.o_draft[step], ref[i].float().cpu().numpy(), f"{name} step {step} req {b}")
            km, vm, kw0, vw0 = mains[b]
            kn, vn = f32(r.k_new[: step + 1]).transpose(1, 0, 2), f32(r.v_new[: step + 1]).transpose(1, 0, 2)
            want = O.draft_attn(f32(r.q[step]), km, vm, np.concatenate([kw0, kn], 1), np.concatenate([vw0, vn], 1))
            assert_attn_close(r.o_draft[step], want, f"{name} step {step} req {b} vs oracle")
        for b in act:
            bt.comp[b].n_win += 1
    # every call leaves the arrival counters at zero (the same kernel runs on the shared array)
    ctr = bt.ws_draft.view(torch.int32)[: vc.VC_DRAFT_COUNTER_BYTES // 4]
    assert int(torch.count_nonzero(ctr).item()) == 0


def test_noalloc_matches_workspace_and_oracle_as_kv_heads_change(vc):
    """tiny (2 KV heads) -> token drop with 8 -> tiny again -> 2-bit with 8: the array holds the
    previous call's partials each time the shape changes."""
    for name in ("tiny", "drop8", "tiny", "quant2"):
        _check_steps(vc, name)


def test_noalloc_rejects_calls_beyond_its_scratch(vc):
    """A shape whose partials exceed the static array is refused with VC_ERR_WORKSPACE, launching nothing."""
    big = vc.vc_shape(32, 1024, 8, 128)
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, big) > vc.VC_DRAFT_NOALLOC_SCRATCH_BYTES
    st = vc.vc_draft_attn_noalloc(big, None, raise_on_error=False, stream=0)
    assert st == vc.VC_ERR_WORKSPACE
