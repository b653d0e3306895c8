"""GPU parity of the integer/byte steps against the oracle, bit for bit: keep-set indices,
quantisation codes/scales/zeros, gathered rows, and accepted tokens/lengths."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import configs, gen
from tests.util import make_batch, f32, assert_quant_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _keepset_case(w, reqs, compact=False):
    bt = make_batch(w, reqs, compact=compact)
    bt.compress()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    for b, r in zip(reqs, bt.reqs):
        ref = O.keep_set(r.importance.cpu().numpy(), w.keep[b], w.recent[b])
        got = r.idx[: len(ref)].cpu().numpy()
        assert np.array_equal(got, ref), f"request {b}: first diff at {np.argmax(got != ref)}"
        assert bt.comp[reqs.index(b)].keep == len(ref)
        if compact:
            kf = r.k_full.cpu()
            assert torch.equal(r.k_rows[:, : len(ref)].cpu(), kf[:, torch.from_numpy(ref).long()])
    return bt


def test_keepset_tiny():
    _keepset_case(configs.tiny(), [0])


def test_keepset_llama8b_full_size():
    """All 8 requests at full size: context 32768, keep 8192 = 512 recent + 7680 by importance."""
    _keepset_case(configs.llama8b_drop(), list(range(8)))


def test_keepset_mixed_contexts_and_compaction():
    w = configs.mixed_serving()
    reqs = w.request_indices("drop")[:6]
    _keepset_case(w, reqs, compact=True)


@pytest.mark.parametrize("n,keep,recent", [(1000, 1000, 0), (1000, 2000, 10), (777, 100, 33), (5000, 1, 0),
                                           (4097, 4096, 0), (3000, 700, 700)])
def test_keepset_edges_with_ties(n, keep, recent):
    """Heavy ties and signed zeros: ties at the threshold go to the lower index."""
    w = configs.scaled(configs.tiny(), batch=1)
    w.ctx, w.keep, w.recent = [n], [keep], [recent]
    bt = make_batch(w, [0])
    rng = np.random.default_rng(n + keep)
    imp = rng.choice(np.array([0.0, -0.0, 0.25, 0.5, 1.0, -3.0], dtype=np.float32), size=n)
    bt.reqs[0].importance.copy_(torch.from_numpy(imp))
    bt.compress()
    torch.cuda.synchronize()
    ref = O.keep_set(imp, keep, recent)
    got = bt.reqs[0].idx[: len(ref)].cpu().numpy()
    assert np.array_equal(got, ref)


def _quant_case(w, reqs):
    bt = make_batch(w, reqs)
    bt.compress()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        assert_quant_state(bt, i, f32(r.k_full), f32(r.v_full), w.bits, w.residual_min)


def test_quant2_qwen_shape_scaled():
    _quant_case(configs.scaled(configs.qwen32b_quant2(), ctx_div=16, batch=3), [0, 1, 2])


def test_quant4_llama70b_shape_scaled():
    _quant_case(configs.scaled(configs.llama70b_offload4(), ctx_div=64, batch=2), [0, 1])


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_d64_ragged_contexts(bits):
    w = configs.scaled(configs.tiny(), batch=3)
    w.mode = ["quant"] * 3
    w.bits = bits
    w.ctx = [1000, 129, 161 + 32 * 7]
    _quant_case(w, [0, 1, 2])


def test_quant2_full_size_one_request():
    """Full Qwen-32B-like context (65536) for one request, every byte."""
    w = configs.qwen32b_quant2()
    _quant_case(w, [0])


# ---------------------------------------------------------------------------- accept -----------
def _accept_case(w, rnd=0, vocab=None):
    draft, logits, L = gen.drafts_and_logits(w, rnd, device="cuda", vocab=vocab)
    from lossless_compressed_kv_vc_gb300 import engine
    tok, nacc = engine.accept(logits, draft, L)
    torch.cuda.synchronize()
    lg, dr = logits.cpu().numpy(), draft.cpu().numpy()
    for b in range(w.B):
        rt, rn = O.accept(lg[b], dr[b], w.L[b])
        assert int(nacc[b]) == rn, f"request {b}"
        got = tok[b].cpu().numpy()
        assert got[:rn].tolist() == rt and np.all(got[rn:] == -1)
    return nacc


def test_accept_tiny():
    _accept_case(configs.tiny())


def test_accept_llama8b_full_size():
    _accept_case(configs.llama8b_drop())


def test_accept_mixed_ragged_L():
    w = configs.mixed_serving()
    _accept_case(w, rnd=3)


def test_accept_edges():
    """All match (bonus), mismatch at 0, ties, L = 0, unaligned vocabulary."""
    from lossless_compressed_kv_vc_gb300 import engine
    for V in (7, 1000, 1001):
        B, Lm = 4, 5
        logits = torch.randn((B, Lm + 1, V), device="cuda")
        logits[2, :, :] = 1.0  # all tied: argmax 0 everywhere
        draft = logits[:, :Lm].argmax(dim=2).to(torch.int32).contiguous()
        draft[1, 0] = (draft[1, 0] + 1) % V
        L = torch.tensor([Lm, Lm, Lm, 0], dtype=torch.int32, device="cuda")
        tok, nacc = engine.accept(logits, draft, L)
        torch.cuda.synchronize()
        lg, dr = logits.cpu().numpy(), draft.cpu().numpy()
        for b in range(B):
            rt, rn = O.accept(lg[b], dr[b], int(L[b]))
            assert int(nacc[b]) == rn and tok[b, :rn].cpu().tolist() == rt
        assert nacc.cpu().tolist() == [Lm + 1, 1, Lm + 1, 1]


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_half_integer_ties(bits):
    """Every key channel and value group spans 0 .. 2^bits - 1 in steps of 1/2 (times a power of two
    per channel), so the scale is exactly a power of two and half the quotients (x - z) / s are
    exact half-integers: the codes must take round-half-even exactly as the oracle does."""
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=256, batch=1)
    w.bits = bits
    w.ctx = [128 + 96]
    bt = make_batch(w, [0])
    r = bt.reqs[0]
    M = 2 * ((1 << bits) - 1) + 1
    t = torch.arange(w.ctx[0], dtype=torch.float32)[:, None]
    c = torch.arange(w.d, dtype=torch.float32)[None, :]
    ramp = torch.remainder(t, M) / 2                            # 0, 0.5, ..., 2^bits - 1
    kv = ramp * torch.pow(2.0, torch.remainder(c, 3) - 1)       # exact in bf16
    vv = (torch.remainder(c + t, M) / 2) * torch.pow(2.0, torch.remainder(t, 3) - 1)
    for h in range(w.Hkv):
        r.k_full[h, : w.ctx[0]].copy_(kv.to(torch.bfloat16))
        r.v_full[h, : w.ctx[0]].copy_(vv.to(torch.bfloat16))
    bt.compress()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    ref = assert_quant_state(bt, 0, f32(r.k_full), f32(r.v_full), bits, w.residual_min)
    assert ref["ng"] == 3


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_flags_scale_out_of_fp16_range(bits):
    """A key channel spanning more than 65504 x (2^bits - 1) in one group has no finite fp16 scale
    (nor, at -6e5, a finite fp16 zero): compress sets VC_DEV_RANGE in the caller's status word."""
    import lossless_compressed_kv_vc_gb300 as vc
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=256, batch=1)
    w.bits = bits
    w.ctx = [224]
    bt = make_batch(w, [0])
    r = bt.reqs[0]
    r.k_full[0, 0, 3] = 6.0e5
    r.k_full[0, 1, 3] = -6.0e5
    bt.dev_status.zero_()
    bt.compress()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == vc.VC_DEV_RANGE
