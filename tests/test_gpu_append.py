"""GPU parity of the post-accept cache update (vc_append_kv) against the oracle.

After an append the caches must hold what compressing the grown context from scratch gives:
KV_full rows, quantised codes, fp16 scales and zeros and the residual window, all bit for bit
against the oracle's quantize_kv of the grown cache, which is built on the host from the seeded
inputs. A two-round case carries one round's accepted drafts into the next round and checks that
round's draft, verify and accept outputs against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import lossless_compressed_kv_vc_gb300 as vc
from workloads import configs, gen
from tests.util import make_batch, f32, assert_attn_close, assert_quant_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()


def _append(bt, rows):
    """One vc_append_kv call; rows[i] = (k, v) bf16 [n][Hkv][d] device tensors for request i."""
    arr = (vc.vc_append_req * len(bt.reqs))()
    for i, (k, v) in enumerate(rows):
        arr[i].n_rows = k.shape[0]
        if k.shape[0] > 0:
            arr[i].k_rows, arr[i].v_rows = k.data_ptr(), v.data_ptr()
    vc.vc_append_kv(bt.shape, bt.full, bt.comp, arr, bt.residual_min, bt.dev_status)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0


def _grown(kf, k_rows):
    """Host float32 cache [Hkv][ctx][d] grown by rows [n][Hkv][d] (token order kept)."""
    return np.concatenate([kf, f32(k_rows).transpose(1, 0, 2)], axis=1)


def _quant_workload(base, bits, ctx):
    w = configs.scaled(base, batch=len(ctx))
    w.mode = ["quant"] * len(ctx)
    w.bits = bits
    w.ctx = list(ctx)
    return w


# Contexts and two successive appends per request. They cover: a residual below residual_min that
# crosses it (157 + 5), no growth at all, a context that stays below residual_min (100 + 7), many
# blocks with one more block (1000 + 40), exactly residual_min + 1 tokens, and the largest staged
# residual (159 + 96 = 255 rows, three new blocks at once).
CTX = [157, 200, 100, 1000, 129, 255]
APPENDS = [[5, 0, 7, 40, 0, 96], [30, 64, 0, 1, 31, 1]]


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("base", ["tiny_d64", "qwen_d128"])
def test_append_quant_equals_compress_of_grown_cache(base, bits):
    w = _quant_workload(configs.tiny() if base == "tiny_d64" else configs.qwen32b_quant2(), bits, CTX)
    grow = max(sum(a[i] for a in APPENDS) for i in range(len(CTX)))
    bt = make_batch(w, list(range(w.B)), grow=grow)
    bt.compress()
    torch.cuda.synchronize()
    host = [(f32(r.k_full[:, : r.ctx]), f32(r.v_full[:, : r.ctx])) for r in bt.reqs]
    for rnd, counts in enumerate(APPENDS, start=1):
        rows = [gen.appended_rows(w, rnd, b, n, "cuda") for b, n in enumerate(counts)]
        _append(bt, rows)
        for i, r in enumerate(bt.reqs):
            kf, vf = _grown(host[i][0], rows[i][0]), _grown(host[i][1], rows[i][1])
            host[i] = (kf, vf)
            assert bt.full[i].ctx == kf.shape[1]
            assert np.array_equal(f32(r.k_full[:, : kf.shape[1]]), kf)
            assert np.array_equal(f32(r.v_full[:, : kf.shape[1]]), vf)
            assert_quant_state(bt, i, kf, vf, bits, w.residual_min)


def test_append_token_drop_grows_full_cache_then_compress_sees_it():
    """Token-drop requests keep their keep-set until the next compress, which then selects from
    the grown context."""
    w = configs.scaled(configs.llama8b_drop(), ctx_div=32, batch=3, L=4)
    bt = make_batch(w, [0, 1, 2], grow=64)
    bt.compress()
    torch.cuda.synchronize()
    keep0 = [bt.comp[i].keep for i in range(3)]
    idx0 = [r.idx.clone() for r in bt.reqs]
    host = [(f32(r.k_full[:, : r.ctx]), f32(r.v_full[:, : r.ctx])) for r in bt.reqs]
    counts = [17, 0, 64]
    rows = [gen.appended_rows(w, 1, b, n, "cuda") for b, n in enumerate(counts)]
    _append(bt, rows)
    for i, r in enumerate(bt.reqs):
        kf, vf = _grown(host[i][0], rows[i][0]), _grown(host[i][1], rows[i][1])
        assert bt.full[i].ctx == w.ctx[i] + counts[i]
        assert np.array_equal(f32(r.k_full[:, : kf.shape[1]]), kf)
        assert np.array_equal(f32(r.v_full[:, : kf.shape[1]]), vf)
        assert bt.comp[i].keep == keep0[i] and torch.equal(r.idx, idx0[i])
    bt.compress()
    torch.cuda.synchronize()
    for i, r in enumerate(bt.reqs):
        ctx2 = w.ctx[i] + counts[i]
        ref = O.keep_set(r.importance[:ctx2].cpu().numpy(), w.keep[i], w.recent[i])
        assert np.array_equal(r.idx[: len(ref)].cpu().numpy(), ref)


def test_append_nothing_is_a_no_op():
    w = _quant_workload(configs.tiny(), 2, [300, 40])
    bt = make_batch(w, [0, 1], grow=8)
    bt.compress()
    torch.cuda.synchronize()
    before = [(r.kc.clone(), r.k_win.clone()) for r in bt.reqs]
    z = torch.empty((0, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
    _append(bt, [(z, z), (z, z)])
    for i, r in enumerate(bt.reqs):
        assert bt.full[i].ctx == w.ctx[i]
        assert torch.equal(r.kc, before[i][0]) and torch.equal(r.k_win, before[i][1])


@pytest.mark.parametrize("mode", ["drop", "quant2", "quant4"])
def test_two_rounds_carry_accepted_drafts(mode):
    """Round 0: compress, draft, verify, accept; append_accepted; round 1 drafts from the grown
    caches (token drop recompresses; quantised caches are used as the append left them) and is
    checked against the oracle on the grown context."""
    if mode == "drop":
        w = configs.scaled(configs.llama8b_drop(), ctx_div=32, batch=3, L=6, vocab=4096)
    else:
        w = configs.scaled(configs.qwen32b_quant2(), ctx_div=64, batch=3, L=6, vocab=4096)
        w.bits = 2 if mode == "quant2" else 4
        w.ctx = [1000, 157, 1100]
    bt = make_batch(w, [0, 1, 2], grow=w.L_max)
    bt.compress()
    bt.prepare_steps()
    B = w.B
    tok = torch.empty((B, w.L_max + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((B,), dtype=torch.int32, device="cuda")
    draft, logits, L = gen.drafts_and_logits(w, 0, device="cuda")
    bt.run_round(logits, draft, L, tok, nacc, compress=False)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    lg, dr = logits.cpu().numpy(), draft.cpu().numpy()
    n_acc = [O.accept(lg[b], dr[b], w.L[b])[1] for b in range(B)]
    assert nacc.cpu().tolist() == n_acc
    host = []
    for i, r in enumerate(bt.reqs):
        n = n_acc[i] - 1
        host.append((_grown(f32(r.k_full[:, : w.ctx[i]]), r.k_new[:n]),
                     _grown(f32(r.v_full[:, : w.ctx[i]]), r.v_new[:n])))
    bt.append_accepted(n_acc)
    # round 1 inputs in place (the descriptors point at these tensors)
    for b, r in enumerate(bt.reqs):
        q, kn, vn = gen.round_queries(w, 1, b, "cuda")
        r.q.copy_(q)
        r.k_new.copy_(kn)
        r.v_new.copy_(vn)
    draft, logits, L = gen.drafts_and_logits(w, 1, device="cuda")
    bt.run_round(logits, draft, L, tok, nacc, compress=(mode == "drop"))
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    lg, dr = logits.cpu().numpy(), draft.cpu().numpy()
    for i, r in enumerate(bt.reqs):
        kf, vf = host[i]
        assert bt.full[i].ctx == kf.shape[1] == r.ctx
        if mode == "drop":
            idx = O.keep_set(r.importance[: kf.shape[1]].cpu().numpy(), w.keep[i], w.recent[i])
            km, vm = O.comp_main_rows("drop", kf, vf, idx=idx)
            kw0 = vw0 = np.zeros((w.Hkv, 0, w.d), np.float32)
        else:
            qkv = O.quantize_kv(kf, vf, w.bits, w.residual_min)
            km, vm = O.comp_main_rows("quant", kf, vf, qkv=qkv)
            kw0, vw0 = qkv["k_res"], qkv["v_res"]
        kn, vn = f32(r.k_new), f32(r.v_new)
        ref_d = O.draft_round(f32(r.q), km, vm, kw0, vw0, kn, vn)
        assert_attn_close(r.o_draft, ref_d, f"round 1 draft, request {i}")
        ref_v = O.verify_attn(f32(r.q), kf, vf, kn.transpose(1, 0, 2), vn.transpose(1, 0, 2))
        assert_attn_close(r.o_verify, ref_v, f"round 1 verify, request {i}")
        rt, rn = O.accept(lg[i], dr[i], w.L[i])
        assert int(nacc[i]) == rn and tok[i, :rn].cpu().tolist() == rt
