"""GPU parity of the SnapKV-style importance (vc_snapkv_importance) against the oracle.

Scores are bf16 products accumulated in fp32 on the tensor cores, the softmax runs in fp32, and a
key's sum over 128 window rows is an MMA of the fp16-rounded weights (relative error <= 2^-11 per
weight, weights <= 1), against the oracle's float64: each element must satisfy
|gpu - oracle| <= 1e-3 |oracle| + 1e-6 max|oracle|. Cases cover 20 to 400 window rows per KV head
(one to four 128-row tiles, ragged), d = 64 and 128, max and average pooling of widths 1, 5 and 7,
contexts that are not tile multiples, a context equal to the window, and full Llama-3-8B-shape
contexts."""
import numpy as np
import pytest
import torch

import oracle as O
import lossless_compressed_kv_vc_gb300 as vc
from workloads import configs, gen
from tests.util import make_batch, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _close(got, ref, what):
    err = np.abs(got - ref)
    lim = 1e-3 * np.abs(ref) + 1e-6 * np.abs(ref).max()
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, worst at {np.argmax(err / lim)}"


def _case(w, reqs, window, pool_kernel=7, pool="max", check_keep=False):
    bt = make_batch(w, reqs)
    q_obs = [gen.observation_queries(w, b, window, "cuda") for b in reqs]
    kind = vc.VC_POOL_MAX if pool == "max" else vc.VC_POOL_AVG
    for r in bt.reqs:
        r.importance.fill_(float("nan"))
    bt.snapkv_importance(q_obs, window, pool_kernel, kind)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        ref = O.snapkv_importance(f32(q_obs[i]), f32(r.k_full[:, : r.ctx]), pool_kernel, pool)
        _close(r.importance[: r.ctx].double().cpu().numpy(), ref, f"{w.name} request {b}")
    if check_keep:  # the keep-set chosen from the GPU importance is the oracle's selection on it
        bt.compress()
        torch.cuda.synchronize()
        for i, b in enumerate(reqs):
            r = bt.reqs[i]
            ref = O.keep_set(r.importance[: r.ctx].cpu().numpy(), w.keep[b], w.recent[b])
            assert np.array_equal(r.idx[: len(ref)].cpu().numpy(), ref)


@pytest.mark.parametrize("window,pool_kernel,pool", [(8, 7, "max"), (16, 5, "avg"), (32, 1, "max"), (64, 7, "avg"),
                                                     (5, 3, "max"), (100, 5, "avg")])
def test_importance_tiny_d64(window, pool_kernel, pool):
    """Tiny workload (d 64, G 4): 32, 64, 128, 256, 20 and 400 window rows per KV head."""
    _case(configs.tiny(), [0], window, pool_kernel, pool)


def test_importance_llama8b_scaled_and_keep_set():
    w = configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=3)
    _case(w, [0, 1, 2], 32, 7, "max", check_keep=True)


@pytest.mark.parametrize("window", [16, 64])
def test_importance_ragged_contexts(window):
    """Contexts off the 64-key tile and 1024-key chunk grid, in one call."""
    w = configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=3)
    w.ctx = [1000, 1025, 3001]
    _case(w, [0, 1, 2], window, 5, "avg")


def test_importance_context_equals_window():
    w = configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=2)
    w.ctx = [32, 33]
    w.keep = [8, 8]
    w.recent = [2, 2]
    _case(w, [0, 1], 32, 3, "max")


def test_importance_llama8b_full_size():
    """Two requests of the full Llama-3-8B-shape workload (context 32768), window 32."""
    _case(configs.llama8b_drop(), [0, 1], 32, 7, "max")


@pytest.mark.parametrize("window", [32, 48])
def test_importance_llama70b_shape_g8(window):
    """64/8 heads (G = 8): 256 or 384 window rows per KV head, i.e. two or three 128-row tiles whose
    column sums are separate partials, d = 128."""
    w = configs.scaled(configs.llama70b_offload4(), ctx_div=64, batch=2)
    w.mode = ["drop", "drop"]
    w.keep = [512, 512]
    w.recent = [32, 32]
    _case(w, [0, 1], window, 7, "max")
