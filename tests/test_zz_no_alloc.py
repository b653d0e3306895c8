"""vc_draft_attn_noalloc: the draft step for callers that cannot allocate device memory (a plugin
whose host application owns all device allocations, or a loop that must not call cudaMalloc).

It is called through the C ABI and must give the same output as vc_draft_attn with a caller
workspace, within the attention tolerance the other tests use, on two calls in a row (the second
call finds the first call's data still in the shared scratch array). This file sorts last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from workloads import configs
from tests.util import make_batch, assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__ as g
    g.build()
    import lossless_compressed_kv_vc_gb300 as m
    return m


@pytest.mark.parametrize("which", ["drop", "quant2"])
def test_noalloc_matches_workspace_entry_point_twice(vc, which):
    if which == "drop":
        w = configs.scaled(configs.llama8b_drop(), ctx_div=8, batch=4, L=2)
    else:
        w = configs.scaled(configs.qwen32b_quant2(), ctx_div=16, batch=3, L=2)
    bt = make_batch(w, list(range(w.B)))
    bt.compress()
    torch.cuda.synchronize()
    lib = vc.lib_handle()
    for step in range(2):  # two calls in a row through the no-allocation entry point
        act, arr = bt.draft_requests(step)
        shape = vc.vc_shape(len(act), w.Hq, w.Hkv, w.d)
        vc.vc_draft_attn(shape, arr, bt.ws_draft, bt.dev_status)
        torch.cuda.synchronize()
        ref = [bt.reqs[b].o_draft[step].clone() for b in act]
        for b in act:
            bt.reqs[b].o_draft[step].fill_(float("nan"))
        st = lib.vc_draft_attn_noalloc(ctypes.byref(shape), arr, ctypes.c_void_p(bt.dev_status.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == vc.VC_OK, vc.vc_status_string(st)
        torch.cuda.synchronize()
        assert int(bt.dev_status.item()) == 0
        for i, b in enumerate(act):
            assert_attn_close(bt.reqs[b].o_draft[step], ref[i].float().cpu().numpy(), f"{which} step {step} req {b}")
        for b in act:
            bt.comp[b].n_win += 1


def test_noalloc_rejects_calls_beyond_its_scratch(vc):
    """A shape whose partials exceed the static array is refused with VC_ERR_WORKSPACE, launching nothing."""
    big = vc.vc_shape(32, 1024, 8, 128)
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, big) > (32 << 20)
    st = vc.vc_draft_attn_noalloc(big, None, raise_on_error=False, stream=0)
    assert st == vc.VC_ERR_WORKSPACE
