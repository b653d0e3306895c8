"""GPU parity at 16 query heads per KV head: the draft kernel's two 8-head blocks per KV head and
verification tiles of 8 drafted rows x 16 heads, against the oracle."""
import pytest
import torch

import oracle as O
from workloads import configs
from tests.util import make_batch, f32, assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _workload(mode, L):
    w = configs.scaled(configs.tiny(), batch=2, L=L)
    w.Hq, w.Hkv = 32, 2
    if mode == "quant":
        w.mode = ["quant"] * 2
        w.bits = 2
        w.ctx = [700, 333]
    return w


@pytest.mark.parametrize("mode", ["drop", "quant"])
def test_draft_sixteen_heads_per_kv_head(mode):
    from tests.test_gpu_draft import _check_all_steps
    _check_all_steps(_workload(mode, 3), [0, 1])


def test_verify_sixteen_heads_per_kv_head():
    w = _workload("drop", 9)  # 9 x 16 = 144 rows: two row tiles per KV head
    bt = make_batch(w, [0, 1])
    for r in bt.reqs:
        r.k_win[:, r.n_res: r.n_res + r.L].copy_(r.k_new.transpose(0, 1))
        r.v_win[:, r.n_res: r.n_res + r.L].copy_(r.v_new.transpose(0, 1))
    bt.verify()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    G = w.Hq // w.Hkv
    for r in bt.reqs:
        q, kf, vf = f32(r.q), f32(r.k_full), f32(r.v_full)
        kn, vn = f32(r.k_new).transpose(1, 0, 2), f32(r.v_new).transpose(1, 0, 2)
        for hk in range(w.Hkv):
            sel = slice(hk * G, (hk + 1) * G)
            ref = O.verify_attn(q[:, sel], kf[hk:hk + 1], vf[hk:hk + 1], kn[hk:hk + 1], vn[hk:hk + 1])
            assert_attn_close(r.o_verify[:, sel], ref, f"G16 hk{hk}")
