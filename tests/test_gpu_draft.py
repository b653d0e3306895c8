"""GPU parity of draft decode attention against the oracle (float tolerance in tests/util.py).

Small cases run every step of every head; full-size cases check sampled (request, head, step)
outputs, which the oracle computes one by one."""
import numpy as np
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


def _run_round(bt, steps=None):
    bt.compress()
    L = max(r.L for r in bt.reqs)
    for s in range(L if steps is None else steps):
        bt.draft_step(s)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0


def _oracle_main(w, b, r, bt_i, bt):
    kf, vf = f32(r.k_full), f32(r.v_full)
    if w.mode[b] == "drop":
        idx = O.keep_set(r.importance.cpu().numpy(), w.keep[b], w.recent[b])
        km, vm = O.comp_main_rows("drop", kf, vf, idx=idx)
        kw0 = np.zeros((w.Hkv, 0, w.d), np.float32)
        vw0 = kw0
    else:
        qkv = O.quantize_kv(kf, vf, w.bits, w.residual_min)
        km, vm = O.comp_main_rows("quant", kf, vf, qkv=qkv)
        kw0, vw0 = qkv["k_res"], qkv["v_res"]
    return km, vm, kw0, vw0


def _check_all_steps(w, reqs, compact=False):
    bt = make_batch(w, reqs, compact=compact)
    _run_round(bt)
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        km, vm, kw0, vw0 = _oracle_main(w, b, r, i, bt)
        ref = O.draft_round(f32(r.q), km, vm, kw0, vw0, f32(r.k_new), f32(r.v_new))
        assert_attn_close(r.o_draft, ref, f"{w.name} request {b}")
        # fused append: the window holds the drafted rows after the round
        assert torch.equal(r.k_win[:, r.n_res: r.n_res + r.L].transpose(0, 1).cpu(), r.k_new.cpu())
        assert torch.equal(r.v_win[:, r.n_res: r.n_res + r.L].transpose(0, 1).cpu(), r.v_new.cpu())


def test_draft_tiny_all_steps():
    _check_all_steps(configs.tiny(), [0])


def test_draft_drop_llama8b_scaled():
    w = configs.scaled(configs.llama8b_drop(), ctx_div=8, batch=3, L=6)
    _check_all_steps(w, [0, 1, 2])


def test_draft_drop_compact():
    w = configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=2, L=4)
    _check_all_steps(w, [0, 1], compact=True)


# kernel: the mma.sync kernel (default) or the tcgen05 one (VC_DRAFT_TC=1); same results
@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_draft_quant2_qwen_scaled(kernel, monkeypatch):
    monkeypatch.setenv("VC_DRAFT_TC", "1" if kernel == "tc" else "0")
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=32, batch=3, L=5)
    _check_all_steps(w, [0, 1, 2])


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_draft_quant4_llama70b_scaled(kernel, monkeypatch):
    monkeypatch.setenv("VC_DRAFT_TC", "1" if kernel == "tc" else "0")
    w = configs.scaled(configs.llama70b_offload4(), ctx_div=128, batch=2, L=5)
    _check_all_steps(w, [0, 1])


@pytest.mark.parametrize("bits", [2, 4])
def test_draft_quant_d64_ragged(bits):
    w = configs.scaled(configs.tiny(), batch=3, L=3)
    w.mode = ["quant"] * 3
    w.bits = bits
    w.ctx = [1000, 140, 2011]
    _check_all_steps(w, [0, 1, 2])


@pytest.mark.parametrize("kernel", ["mma", "tc"])
@pytest.mark.parametrize("bits", [2, 4])
def test_draft_quant_d128_ragged(kernel, bits, monkeypatch):
    """d = 128, G = 5, contexts that leave 0, 1, 3, 5 and 61 quantised groups (a window-only
    request; partial four-group blocks of the tcgen05 kernel; residuals of 128-150 rows, window
    blocks of up to 156 rows): most CTAs of a KV head's grid row hold a little of a request, some
    none, so the split partials and their merge are exercised with empty slots."""
    monkeypatch.setenv("VC_DRAFT_TC", "1" if kernel == "tc" else "0")
    w = configs.scaled(configs.qwen32b_quant2(), batch=5, L=6)
    w.bits = bits
    w.ctx = [150, 160, 224, 300, 2100]
    _check_all_steps(w, [0, 1, 2, 3, 4])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vscale", [1e-3, 300.0])
def test_draft_quant_value_scales(bits, vscale):
    """Value caches far from unit size (every value times 1e-3 or 300, then bf16): the quantised
    kernel's fp16 operands -- value scales and zeros, weights times scales (for 2 bits with a
    factor 1/16 on half the tokens), codes as fp16 subnormals -- against the oracle on every step.
    Both sides are divided by the factor before the comparison: the outputs scale with the values,
    and so does every rounding error, while the tolerance's absolute floor (1e-2) is set for
    outputs of unit size."""
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=64, batch=2, L=4)
    w.bits = bits
    reqs = [0, 1]
    bt = make_batch(w, reqs)
    for r in bt.reqs:
        r.v_full.copy_((r.v_full.float() * vscale).to(torch.bfloat16))
        r.v_new.copy_((r.v_new.float() * vscale).to(torch.bfloat16))
    _run_round(bt)
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        km, vm, kw0, vw0 = _oracle_main(w, b, r, i, bt)
        ref = O.draft_round(f32(r.q), km, vm, kw0, vw0, f32(r.k_new), f32(r.v_new))
        assert_attn_close(r.o_draft.float() / vscale, ref / vscale, f"{w.name} request {b} values x {vscale}")


@pytest.mark.parametrize("keep,ctx,L", [(10, 64, 3), (17, 40, 17), (1, 8, 2)])
def test_draft_fewer_chunks_than_warps(keep, ctx, L):
    """One request whose step has only 2-3 chunks per head (16-row kept chunks, then window
    chunks): a one-CTA launch where some warps hold no chunk; the split partials of the request
    must be merged from the warps that hold it only."""
    w = configs.scaled(configs.tiny(), batch=1, L=L)
    w.ctx, w.keep, w.recent = [ctx], [keep], [0]
    _check_all_steps(w, [0])


def test_draft_keep_all_equals_full_attention_on_gpu():
    """keep = ctx: the draft output equals attention over the whole cache (NS invariant)."""
    w = configs.scaled(configs.tiny(), batch=2, L=3)
    w.keep = [w.ctx[0]] * 2
    bt = make_batch(w, [0, 1])
    _run_round(bt)
    for i in range(2):
        r = bt.reqs[i]
        ref = O.verify_attn(f32(r.q), f32(r.k_full), f32(r.v_full), f32(r.k_new).transpose(1, 0, 2),
                            f32(r.v_new).transpose(1, 0, 2))
        assert_attn_close(r.o_draft, ref, "keep-all")


def _sampled_full_size(w, reqs, steps, heads):
    bt = make_batch(w, reqs)
    _run_round(bt)
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        km, vm, kw0, vw0 = _oracle_main(w, b, r, i, bt)
        q, kn, vn = f32(r.q), f32(r.k_new), f32(r.v_new)
        G = w.Hq // w.Hkv
        for s in steps:
            kw = np.concatenate([kw0, kn[: s + 1].transpose(1, 0, 2)], axis=1)
            vw = np.concatenate([vw0, vn[: s + 1].transpose(1, 0, 2)], axis=1)
            for hk in heads:
                sel = slice(hk * G, (hk + 1) * G)
                ref = O.draft_attn(q[s, sel], km[hk:hk + 1], vm[hk:hk + 1], kw[hk:hk + 1], vw[hk:hk + 1])
                assert_attn_close(r.o_draft[s, sel], ref, f"{w.name} b{b} s{s} hk{hk}")


def test_draft_llama8b_full_size_sampled():
    w = configs.llama8b_drop()
    _sampled_full_size(w, list(range(8)), steps=[0, 31], heads=[0, 7])


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_draft_qwen32b_quant2_full_size_sampled(kernel, monkeypatch):
    monkeypatch.setenv("VC_DRAFT_TC", "1" if kernel == "tc" else "0")
    w = configs.qwen32b_quant2()
    _sampled_full_size(w, [0, 15] + list(range(1, 15)), steps=[0, 24], heads=[3])


@pytest.mark.parametrize("bad", ["past_end", "negative"])
def test_draft_flags_out_of_range_keep_index(bad):
    """A keep-set index at or past KV_full's rows, or a negative one, is not read: the draft step
    sets VC_DEV_BOUNDS in the caller's status word, a kept row of the same chunk stands in, and
    the outputs stay finite."""
    import lossless_compressed_kv_vc_gb300 as vc
    w = configs.scaled(configs.llama8b_drop(), ctx_div=32, batch=1, L=2)
    bt = make_batch(w, [0])
    bt.compress()
    torch.cuda.synchronize()
    r = bt.reqs[0]
    r.idx[7] = w.ctx[0] + 10 if bad == "past_end" else -3
    bt.dev_status.zero_()
    bt.reset_window()
    bt.draft_step(0)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == vc.VC_DEV_BOUNDS
    assert torch.isfinite(r.o_draft[0].float()).all()
