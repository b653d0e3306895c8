"""Pins of the CPU oracle to facts fixed outside it: closed forms, brute force on tiny inputs,
textbook library routines and invariants. Each test names the mistake it is there to catch.

The method is "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", section
"Core algorithm" (draft on KV_comp, verify on KV_full in one pass, accept to the first mismatch
plus a bonus token) and "Architecture support" (token-drop and quantising compressors).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from workloads import gen, configs


# ---------------------------------------------------------------- attention ---------------------
def test_attention_two_key_closed_form(golden_dir):
    """Scores (1, 0) give weights e/(e+1), 1/(e+1). Catches a dropped or wrong 1/sqrt(d) scale
    (1/d would give weights from scores (0.5, 0)) and a missing normalisation."""
    c = json.load(open(os.path.join(golden_dir, "attention_two_key.json")))
    w1 = math.e / (math.e + 1.0)
    v = np.array(c["v"])
    expected = w1 * v[0] + (1.0 - w1) * v[1]
    got = O.attention(np.array([c["q"]]), np.array(c["k"]), v)[0]
    np.testing.assert_allclose(got, expected, rtol=0, atol=1e-14)


def test_attention_equal_keys_gives_mean_of_values():
    """All scores equal -> uniform weights -> mean of V. Catches weights not summing to one."""
    rng = np.random.default_rng(1)
    k = np.tile(rng.standard_normal(16), (37, 1))
    v = rng.standard_normal((37, 16))
    q = rng.standard_normal((3, 16))
    got = O.attention(q, k, v)
    np.testing.assert_allclose(got, np.tile(v.mean(axis=0), (3, 1)), atol=1e-13)


def test_attention_dominant_score_selects_row():
    """One score 60 above the rest selects its value row. Catches transposed score indexing."""
    d = 8
    k = np.zeros((5, d)); k[3, 0] = 60.0 * math.sqrt(d) / 2.0
    q = np.zeros((1, d)); q[0, 0] = 2.0
    v = np.arange(5 * d, dtype=np.float64).reshape(5, d)
    np.testing.assert_allclose(O.attention(q, k, v)[0], v[3], atol=1e-20 + 1e-12)


def test_attention_brute_force_tiny():
    """Explicit per-element loops with math.exp, no max subtraction, on a tiny case."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 4)); k = rng.standard_normal((5, 4)); v = rng.standard_normal((5, 3))
    ref = np.zeros((2, 3))
    for i in range(2):
        w = [math.exp(sum(q[i, c] * k[j, c] for c in range(4)) / 2.0) for j in range(5)]
        z = sum(w)
        for c in range(3):
            ref[i, c] = sum(w[j] * v[j, c] for j in range(5)) / z
    np.testing.assert_allclose(O.attention(q, k, v), ref, atol=1e-13)


def test_attention_mask_excludes_keys():
    """A masked key carries no weight: masking the dominant key falls back to the others."""
    k = np.array([[10.0, 0], [0, 0], [0, 0]]); v = np.array([[100.0, 0], [1.0, 0], [3.0, 0]])
    q = np.array([[1.0, 0]])
    vis = np.array([[False, True, True]])
    np.testing.assert_allclose(O.attention(q, k, v, vis)[0], [2.0, 0.0], atol=1e-14)


def test_attention_permutation_invariant():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 16)); k = rng.standard_normal((50, 16)); v = rng.standard_normal((50, 16))
    p = rng.permutation(50)
    np.testing.assert_allclose(O.attention(q, k, v), O.attention(q, k[p], v[p]), atol=1e-13)


def test_draft_gqa_head_mapping():
    """Query head h reads KV head h // G: values constant per KV head make the output h//G + 1.
    Catches h % Hkv (which differs whenever G > 1 and Hkv > 1)."""
    Hq, Hkv, d = 8, 2, 4
    rng = np.random.default_rng(4)
    q = rng.standard_normal((Hq, d))
    km = rng.standard_normal((Hkv, 6, d)); vm = np.zeros((Hkv, 6, d))
    kw = rng.standard_normal((Hkv, 2, d)); vw = np.zeros((Hkv, 2, d))
    for j in range(Hkv):
        vm[j] = j + 1; vw[j] = j + 1
    out = O.draft_attn(q, km, vm, kw, vw)
    for h in range(Hq):
        np.testing.assert_allclose(out[h], np.full(d, h // (Hq // Hkv) + 1.0), atol=1e-14)


def test_verify_causal_closed_form():
    """Zero keys -> uniform weights over the visible rows. With V_full = 0 and new value row j
    equal to (j+1), row i's output is (i+1)(i+2)/2 / (ctx+i+1). Catches an off-by-one in the
    causal mask (j < i or j <= i+1) and a wrong ctx offset."""
    Hq, Hkv, d, ctx, n = 4, 2, 4, 7, 5
    q = np.random.default_rng(5).standard_normal((n, Hq, d))
    kf = np.zeros((Hkv, ctx, d)); vf = np.zeros((Hkv, ctx, d))
    kn = np.zeros((Hkv, n, d)); vn = np.zeros((Hkv, n, d))
    for j in range(n):
        vn[:, j, :] = j + 1
    out = O.verify_attn(q, kf, vf, kn, vn)
    for i in range(n):
        np.testing.assert_allclose(out[i], (i + 1) * (i + 2) / 2 / (ctx + i + 1), atol=1e-14)


def _small_request(seed=0):
    w = configs.scaled(configs.llama8b_drop(), ctx_div=256, batch=1, L=5)
    w.Hq, w.Hkv, w.d = 8, 2, 32
    r = gen.request(w, 0, 0)
    return w, r


def test_verify_row_equals_decode_at_its_position():
    """Verify row i equals single-token decode at position ctx+i over KV_full + new rows 0..i."""
    w, r = _small_request()
    kf, vf = O.bf16_to_f32(r.k_full), O.bf16_to_f32(r.v_full)
    q = O.bf16_to_f32(r.q); kn = O.bf16_to_f32(r.k_new); vn = O.bf16_to_f32(r.v_new)
    ver = O.verify_attn(q, kf, vf, kn.transpose(1, 0, 2), vn.transpose(1, 0, 2))
    for i in range(q.shape[0]):
        dec = O.draft_attn(q[i], kf, vf, kn[: i + 1].transpose(1, 0, 2), vn[: i + 1].transpose(1, 0, 2))
        np.testing.assert_allclose(ver[i], dec, atol=1e-12)


def test_draft_keep_all_equals_full_attention():
    """Token drop keeping every token makes draft step s equal verify row s."""
    w, r = _small_request()
    kf, vf = O.bf16_to_f32(r.k_full), O.bf16_to_f32(r.v_full)
    q = O.bf16_to_f32(r.q); kn = O.bf16_to_f32(r.k_new); vn = O.bf16_to_f32(r.v_new)
    idx = O.keep_set(O.bf16_to_f32(r.importance), w.ctx[0], 0)
    assert np.array_equal(idx, np.arange(w.ctx[0]))
    km, vm = O.comp_main_rows("drop", kf, vf, idx=idx)
    H = kf.shape[0]
    dr = O.draft_round(q, km, vm, np.zeros((H, 0, w.d)), np.zeros((H, 0, w.d)), kn, vn)
    ver = O.verify_attn(q, kf, vf, kn.transpose(1, 0, 2), vn.transpose(1, 0, 2))
    np.testing.assert_allclose(dr, ver, atol=1e-12)


# ---------------------------------------------------------------- keep-set ---------------------
def _keep_brute(imp, keep, recent):
    n = len(imp)
    if keep >= n:
        return list(range(n))
    cand = sorted(range(n - recent), key=lambda i: (-float(imp[i]), i))[: keep - recent]
    return sorted(cand + list(range(n - recent, n)))


@pytest.mark.parametrize("n,keep,recent", [(1, 1, 0), (10, 3, 0), (64, 16, 4), (300, 77, 77),
                                           (4096, 1024, 128), (100, 100, 10), (50, 200, 5), (257, 1, 0)])
def test_keep_set_matches_sorted_brute_force(n, keep, recent):
    """Python sorted() with key (-importance, index) on values with many ties and signed zeros.
    Catches ties to the higher index, a recent window taken from the candidates, unsorted output."""
    rng = np.random.default_rng(n + keep)
    imp = rng.choice(np.array([0.0, -0.0, 0.25, 0.5, 1.0, -3.0], dtype=np.float32), size=n)
    got = O.keep_set(imp, keep, recent)
    assert got.dtype == np.int32
    assert got.tolist() == _keep_brute(imp, keep, recent)


def test_keep_set_uniform_importance_distinct():
    imp = np.random.default_rng(9).random(2000, dtype=np.float32)
    got = O.keep_set(imp, 500, 50)
    assert len(got) == 500 and np.all(np.diff(got) > 0)
    assert np.array_equal(got[-50:], np.arange(1950, 2000))
    thr = np.sort(imp[:1950])[::-1][449]
    assert np.all(imp[got[:-50]] >= thr)


# ---------------------------------------------------------------- quantisation -----------------
@pytest.mark.parametrize("bits", [2, 4])
def test_quant_constant_group(bits):
    """A constant group has scale 0: all codes 0 and x_hat = z exactly."""
    x = np.full((3, 32), 1.3125, dtype=np.float32)
    c, s, z = O.quant_groups(x, bits)
    assert np.all(c == 0) and np.all(s == 0) and np.all(z == np.float16(1.3125))


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_exact_grid(bits):
    """Values on an exactly representable grid z + c*s map to c, with min -> 0 and max -> 2^b-1."""
    qmax = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, qmax + 1, size=32); codes[0] = 0; codes[1] = qmax
    x = (-1.0 + 0.5 * codes).astype(np.float32)[None, :]
    c, s, z = O.quant_groups(x, bits)
    assert s[0] == np.float16(0.5) and z[0] == np.float16(-1.0)
    assert np.array_equal(c[0], codes)


def test_quant_round_half_even():
    """(x - z)/s = 0.5, 1.5, 2.5 exactly -> codes 0, 2, 2 (half to even); half-up would give 1, 2, 3."""
    x = np.zeros(32, dtype=np.float32); x[1] = 3.0; x[2] = 0.5; x[3] = 1.5; x[4] = 2.5
    c, s, z = O.quant_groups(x[None], 2)
    assert s[0] == 1.0 and z[0] == 0.0
    assert c[0, :5].tolist() == [0, 3, 0, 2, 2]


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_error_bound_random(bits):
    """|x - x_hat| <= s/2 plus the fp16 rounding of z and s (relative 2^-11 each, times the codes)."""
    rng = np.random.default_rng(7 + bits)
    x = (rng.standard_normal((500, 32)) * rng.uniform(0.01, 10, size=(500, 1))).astype(np.float32)
    c, s, z = O.quant_groups(x, bits)
    s32, z32 = s.astype(np.float32)[:, None], z.astype(np.float32)[:, None]
    xh = c.astype(np.float32) * s32 + z32
    qmax = (1 << bits) - 1
    bound = s32 / 2 + np.abs(z32) * 2.0 ** -11 + qmax * s32 * 2.0 ** -11 + np.abs(x) * 2.0 ** -20 + 1e-30
    assert np.all(np.abs(x - xh) <= bound * (1 + 1e-6))
    assert np.all(c <= qmax)


def test_fp16_rne_matches_torch_half():
    """fp16 conversion against torch's independent implementation, including ties and subnormals."""
    vals = np.array([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 65504.0, 65519.0, 2.0 ** -24,
                     3 * 2.0 ** -26, 0.1, -0.333, 1e-8, 2.0 ** -25], dtype=np.float32)
    ref = torch.from_numpy(vals).half().numpy()
    got = O.fp16_rne(vals)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_pack_golden(golden_dir):
    cs = json.load(open(os.path.join(golden_dir, "pack_cases.json")))["cases"]
    for c in cs:
        got = O.pack(np.array(c["codes"], dtype=np.uint8), c["bits"])
        assert got.tolist() == c["bytes"], c
        assert O.unpack(got, c["bits"]).tolist() == c["codes"]


@pytest.mark.parametrize("bits", [2, 4])
def test_quant_group_axes(bits):
    """Keys group 32 tokens per channel, values 32 channels per token: an outlier at (t=5, c=7)
    changes only key scale (group 0, channel 7) and only value scale (token 5, channel group 0).
    Catches transposed group axes."""
    rng = np.random.default_rng(11)
    H, ctx, d = 2, 128 + 64, 64
    k = rng.standard_normal((H, ctx, d)).astype(np.float32); v = k.copy()
    base = O.quantize_kv(k, v, bits)
    k2 = k.copy(); v2 = v.copy(); k2[1, 5, 7] = 50.0; v2[1, 5, 7] = 50.0
    q2 = O.quantize_kv(k2, v2, bits)
    dk = np.argwhere(base["ks"] != q2["ks"]); dv = np.argwhere(base["vs"] != q2["vs"])
    assert dk.tolist() == [[1, 0, 7]]
    assert dv.tolist() == [[1, 5, 0]]


def test_quant_layout_rule():
    assert O.quant_layout(65536) == (2044, 128)
    assert O.quant_layout(131072) == (4092, 128)
    assert O.quant_layout(1000) == (27, 136)
    assert O.quant_layout(100) == (0, 100)
    for ctx in range(128, 400):
        ng, nr = O.quant_layout(ctx)
        assert 128 <= nr < 160 and 32 * ng + nr == ctx


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_dequantize_roundtrip(bits):
    rng = np.random.default_rng(12)
    H, ctx, d = 2, 300, 64
    k = rng.standard_normal((H, ctx, d)).astype(np.float32); v = rng.standard_normal((H, ctx, d)).astype(np.float32)
    qkv = O.quantize_kv(k, v, bits)
    ng, nr = O.quant_layout(ctx)
    assert qkv["kc"].shape == (H, ng, 32 * d * bits // 8) and qkv["vc"].shape == (H, ng, 32 * d * bits // 8)
    assert qkv["ks"].shape == (H, ng, d) and qkv["vs"].shape == (H, 32 * ng, d // 32)
    kh, vh = O.dequantize_kv(qkv, d)
    tol = {2: 1.6, 4: 0.35}[bits]
    assert np.abs(kh - k[:, :32 * ng]).max() < tol and np.abs(vh - v[:, :32 * ng]).max() < tol
    assert np.array_equal(qkv["k_res"], k[:, 32 * ng:])


def _grid_cache(bits, H=2, ng=3, d=64, seed=5):
    """K and V [H][32 ng + 128][d] whose every quantisation group lies on its own grid z + c s, with
    s and z exact in fp16, distinct per group, and codes 0 and 2^b - 1 both present, so that
    quantize_kv finds exactly (s, z, c) and the dequantised values equal the inputs bit for bit.
    Keys group 32 tokens per (block, channel), values 32 channels per token. Returns (k, v, key
    codes [H][Tq][d], value codes [H][Tq][d])."""
    rng = np.random.default_rng(seed)
    qmax = (1 << bits) - 1
    Tq, ctx = 32 * ng, 32 * ng + 128

    def grid(n_groups):
        c = rng.integers(0, qmax + 1, size=(n_groups, 32))
        for g in range(n_groups):
            a, b = rng.choice(32, size=2, replace=False)
            c[g, a], c[g, b] = 0, qmax
        s = rng.integers(1, 64, size=(n_groups, 1)) * 2.0 ** -6    # 1/64 .. 63/64, exact in fp16
        z = rng.integers(-256, 256, size=(n_groups, 1)) * 2.0 ** -7  # exact in fp16
        return c, (z + c * s).astype(np.float32)

    kc, kx = grid(H * ng * d)                      # groups (h, block, channel) x 32 tokens
    k = np.zeros((H, ctx, d), np.float32)
    k[:, :Tq] = kx.reshape(H, ng, d, 32).transpose(0, 1, 3, 2).reshape(H, Tq, d)
    vc, vx = grid(H * Tq * (d // 32))              # groups (h, token, channel group) x 32 channels
    v = np.zeros((H, ctx, d), np.float32)
    v[:, :Tq] = vx.reshape(H, Tq, d)
    k[:, Tq:] = rng.standard_normal((H, 128, d)).astype(np.float32)
    v[:, Tq:] = rng.standard_normal((H, 128, d)).astype(np.float32)
    kcodes = kc.reshape(H, ng, d, 32).transpose(0, 1, 3, 2).reshape(H, Tq, d)
    return k, v, kcodes, vc.reshape(H, Tq, d)


@pytest.mark.parametrize("bits", [2, 4])
def test_dequantize_exact_on_grid(bits):
    """Groups on an exact grid come back bit for bit through quantize_kv -> dequantize_kv (every
    code, scale and zero is exact, so x_hat = c s + z reproduces x). Catches a dequantiser that adds
    half a step, swaps the scale and zero of neighbouring groups, or reads the words in another
    order: every group has its own s and z, and codes 0 and 2^b - 1 both occur."""
    k, v, kcodes, vcodes = _grid_cache(bits)
    qkv = O.quantize_kv(k, v, bits)
    ng, Tq = qkv["ng"], 32 * qkv["ng"]
    assert ng == 3
    assert np.array_equal(O.unpack_block(qkv["kc"], bits, "k", 64).reshape(2, Tq, 64), kcodes)
    assert np.array_equal(O.unpack_block(qkv["vc"], bits, "v", 64).reshape(2, Tq, 64), vcodes)
    kh, vh = O.dequantize_kv(qkv, 64)
    assert kh.dtype == np.float32 and vh.dtype == np.float32
    assert np.array_equal(kh, k[:, :Tq]) and np.array_equal(vh, v[:, :Tq])


@pytest.mark.parametrize("bits", [2, 4])
def test_dequantize_error_bound(bits):
    """|x - dequantize_kv(quantize_kv(x))| <= s/2 plus the fp16 rounding of s and z, computed
    through dequantize_kv itself, with each element's own group scale: key (h, block, channel),
    value (h, token, channel group). A half-step offset breaks the bound on about half the
    elements."""
    rng = np.random.default_rng(31 + bits)
    H, d, ng = 2, 64, 5
    ctx = 32 * ng + 128
    k = (rng.standard_normal((H, ctx, d)) * rng.uniform(0.05, 8, size=(H, 1, d))).astype(np.float32)
    v = (rng.standard_normal((H, ctx, d)) * rng.uniform(0.05, 8, size=(H, ctx, 1))).astype(np.float32)
    qkv = O.quantize_kv(k, v, bits)
    kh, vh = O.dequantize_kv(qkv, d)
    Tq, qmax = 32 * ng, (1 << bits) - 1
    ks = np.repeat(qkv["ks"].astype(np.float32), 32, axis=1)          # [H][Tq][d]: block of the token
    kz = np.repeat(qkv["kz"].astype(np.float32), 32, axis=1)
    vs = np.repeat(qkv["vs"].astype(np.float32), 32, axis=2)          # [H][Tq][d]: group of the channel
    vz = np.repeat(qkv["vz"].astype(np.float32), 32, axis=2)
    for x, xh, s, z in ((k[:, :Tq], kh, ks, kz), (v[:, :Tq], vh, vs, vz)):
        bound = s / 2 + np.abs(z) * 2.0 ** -11 + qmax * s * 2.0 ** -11 + np.abs(x) * 2.0 ** -20
        assert np.all(np.abs(x - xh) <= bound * (1 + 1e-6))
        # and the bound is not loose: some element sits near half a step from its value
        assert np.max(np.abs(x - xh) / s) > 0.4


# ---------------------------------------------------------------- accept -----------------------
def test_accept_golden(golden_dir):
    cs = json.load(open(os.path.join(golden_dir, "accept_cases.json")))["cases"]
    for c in cs:
        tok, n = O.accept(np.array(c["logits"], dtype=np.float32), c["draft"], c["L"])
        assert tok == c["tokens"] and n == c["n_acc"], c["name"]


def test_accept_all_match_gives_L_plus_one():
    rng = np.random.default_rng(13)
    L, V = 6, 50
    lg = rng.standard_normal((L + 1, V)).astype(np.float32)
    x = lg[:L].argmax(axis=1)
    tok, n = O.accept(lg, x, L)
    assert n == L + 1 and tok == list(x) + [int(lg[L].argmax())]


def test_accept_mismatch_at_zero_gives_one():
    rng = np.random.default_rng(14)
    L, V = 6, 50
    lg = rng.standard_normal((L + 1, V)).astype(np.float32)
    x = lg[:L].argmax(axis=1); x[0] = (x[0] + 1) % V
    tok, n = O.accept(lg, x, L)
    assert n == 1 and tok == [int(lg[0].argmax())]


def test_planted_logits_mean_accept_length():
    """Planted matches are independent with probability p, so E[n_acc] = (1 - p^(L+1)) / (1 - p).
    Pins the input recipe and accept together (a wrong bonus rule shifts the mean by ~p^L)."""
    w = configs.scaled(configs.tiny(), batch=400)
    w.V = 64
    draft, logits, L = gen.drafts_and_logits(w, 0)
    ns = [O.accept(logits[b].numpy(), draft[b].tolist(), int(L[b]))[1] for b in range(w.B)]
    p, Lb = w.p[0], w.L[0]
    mean = (1 - p ** (Lb + 1)) / (1 - p)
    var = sum((2 * i + 1) * p ** i for i in range(1, Lb + 1)) + 1 - mean ** 2
    assert abs(np.mean(ns) - mean) < 4 * math.sqrt(var / w.B)


def test_block_layout_hand_derived_words():
    """One nonzero code per block, its word and bit worked out by hand from the layout rule:
    keys  (4-bit, d=32): code 5 at (token 9, channel 3): token 9 = 8 + lane//4 -> lane//4 = 1,
          channel 3 = 2*(lane%4) + 1 -> lane%4 = 1, so lane 5, pair 1 (rows +8) high code, bits 20..23
          of word [half 0][j 0][lane 5] = word 5.
    keys  (2-bit, d=32): code 3 at (token 2, channel 17): lane//4 = 2, 17 = 16 + 2*0 + 1 -> lane 8,
          step j = 1 = 2*0 + 1 -> pair f = 4 + 0, high code at bits 16 + 8 = 24 of word [0][0][8] = word 8.
    values(4-bit, d=32): code 7 at (token 17, channel 10): token 17 = 16*1 + 2*0 + 1 -> half 1,
          lane%4 = 0, high code; channel 10 = 8 + 2 -> lane//4 = 2, pair 1 -> bits 20..23 of word
          [half 1][j 0][lane 8] = word (1*2 + 0)*32 + 8 = 72.
    Catches a transposed pair order, a swapped half or lane mapping, and wrong bit offsets."""
    cases = [(4, "k", 9, 3, 5, 5, 20), (2, "k", 2, 17, 3, 8, 24), (4, "v", 17, 10, 7, 72, 20)]
    for bits, kind, t, c, code, word, bit in cases:
        codes = np.zeros((32, 32), dtype=np.uint8)
        codes[t, c] = code
        w = O.pack_block(codes, bits, kind).view("<u4")
        expect = np.zeros_like(w)
        expect[word] = code << bit
        assert np.array_equal(w, expect), (bits, kind, np.nonzero(w), w[np.nonzero(w)])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kind", ["k", "v"])
def test_block_layout_is_a_permutation(bits, kind):
    """Every (token, channel) of a block appears exactly once, and unpack inverts pack."""
    d = 128
    pos = O.frag_positions(d, kind).reshape(-1, 2)
    assert len({tuple(x) for x in pos}) == 32 * d
    codes = np.random.default_rng(bits).integers(0, 1 << bits, size=(2, 32, d)).astype(np.uint8)
    assert np.array_equal(O.unpack_block(O.pack_block(codes, bits, kind), bits, kind, d), codes)


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_with_no_whole_block(bits):
    """ctx < 128 + 32 leaves no whole quantised block: everything stays in the bf16 residual."""
    rng = np.random.default_rng(21)
    k = rng.standard_normal((2, 140, 64)).astype(np.float32)
    qkv = O.quantize_kv(k, k, bits)
    assert qkv["ng"] == 0 and qkv["kc"].shape == (2, 0, 32 * 64 * bits // 8)
    assert np.array_equal(qkv["k_res"], k)
    kh, vh = O.dequantize_kv(qkv, 64)
    assert kh.shape == (2, 0, 64) and vh.shape == (2, 0, 64)


# ---------------------------------------------------------------------------- staggering plan --
def _simulate_streams(costs, groups, periods=1680):
    """Run the two streams of the stagger for many periods, event by event: the copy stream copies
    group 1 then group 0, each copy waiting for the previous verification of its group (its
    staging slot); the compute stream drafts group 0, verifies group 1 (after that period's copy of
    group 1), drafts group 1, verifies group 0 (after its copy). Returns twice the mean period over
    the second half (840 periods: a multiple of every cyclicity a six-event system can have)."""
    from fractions import Fraction
    tot = lambda g, i: sum(c[i] for c, x in zip(costs, groups) if x == g)
    d0, v0, s0 = tot(0, 0), tot(0, 1), tot(0, 2)
    d1, v1, s1 = tot(1, 0), tot(1, 1), tot(1, 2)
    compute = copy = ver0 = ver1 = 0
    ends = []
    for _ in range(periods):
        c1 = max(copy, ver1) + s1
        c0 = max(c1, ver0) + s0
        copy = c0
        t = compute + d0
        t = max(t, c1) + v1
        ver1 = t
        t = t + d1
        t = max(t, c0) + v0
        ver0 = t
        compute = t
        ends.append(t)
    h = periods // 2
    return Fraction(2 * (ends[-1] - ends[h - 1]), periods - h)


def test_stagger_period_matches_stream_simulation():
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 7))
        costs = [tuple(int(x) for x in rng.integers(0, 50, 3)) for _ in range(n)]
        groups = [int(x) for x in rng.integers(0, 2, n)]
        assert O.stagger_period2(costs, groups) == _simulate_streams(costs, groups)


def test_stagger_copy_bound_pairs_split():
    """Two requests each copying 100 and verifying 50, no drafting: together in one group the copy
    and its verification chain (S_0 + V_0 = 300); split, the copy stream bounds it (S = 200)."""
    groups, t = O.plan_stagger([(0, 50, 100), (0, 50, 100)])
    assert groups == [0, 1] and t == 200
    assert O.stagger_period([(0, 50, 100), (0, 50, 100)], [0, 0]) == 300


def test_stagger_balanced_split_unique_size():
    """Four requests (d 0, v 10, s 10): k of them in group 0 give max(40, 40, 20k, 20(4 - k), 40,
    40), least (40) only at k = 2; the smallest mask with two of requests 1..3 in group 1 is 0b011."""
    groups, t = O.plan_stagger([(0, 10, 10)] * 4)
    assert groups == [0, 1, 1, 0] and t == 40


def test_stagger_resident_only_any_split():
    """No copies: every split costs D + V = 32, so the phase work max(D_0 + V_1, D_1 + V_0) decides.
    Worked by hand over the 7 splits: group 1 = {3} gives max(15 + 0, 11 + 6) = 17, {2, 3} gives
    max(12 + 3, 14 + 3) = 17, every other split more (request 1 alone: max(19 + 1, 7 + 5) = 20); of
    the two, the smaller mask 0b100 (request 3). A single request stays alone in group 0: its copy
    overlaps its own drafting and its verification follows the copy, max(D, S) + V = 11."""
    costs = [(5, 2, 0), (7, 1, 0), (3, 3, 0), (11, 0, 0)]
    groups, t = O.plan_stagger(costs)
    assert t == 26 + 6 and groups == [0, 0, 0, 1]
    assert O.stagger_phase_work(costs, groups) == 17
    assert O.stagger_phase_work(costs, [0, 1, 0, 0]) == 20 and O.stagger_phase_work(costs, [0, 0, 1, 1]) == 17
    assert O.plan_stagger([(5, 2, 9)]) == ([0], 11)


def test_stagger_bounds_and_symmetry():
    rng = np.random.default_rng(3)
    for _ in range(100):
        n = int(rng.integers(1, 8))
        costs = [tuple(int(x) for x in rng.integers(0, 100, 3)) for _ in range(n)]
        D, V, S = (sum(c[i] for c in costs) for i in range(3))
        groups, t = O.plan_stagger(costs)
        assert max(D + V, S) <= t <= D + S + V
        assert O.stagger_period2(costs, [1 - g for g in groups]) == O.stagger_period2(costs, groups)


# ---------------------------------------------------------------------------- SnapKV importance --
def test_snapkv_votes_sum_to_rows():
    """Every (window query, head) row is a softmax over its visible keys: the votes sum to W * Hq."""
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal((6, 8, 16)), rng.standard_normal((2, 50, 16))
    assert math.isclose(O.snapkv_votes(q, k).sum(), 6 * 8, rel_tol=1e-12)


def test_snapkv_single_query_is_attention_weights():
    """W = 1, one head: the votes are the last query's attention weights, i.e. the (pinned)
    attention of that query over the keys with one-hot values."""
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 40, 16))
    ref = O.attention(q[0], k[0], np.eye(40))[0]
    assert np.allclose(O.snapkv_votes(q, k), ref, rtol=1e-12, atol=1e-15)


def test_snapkv_constant_keys_closed_form():
    """Identical keys make every row uniform over its visible keys: with ctx = 10 and W = 3, query i
    sees keys 0 .. 7 + i, so vote[t] = Hq * sum over i with t <= 7 + i of 1 / (8 + i)."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 4, 8))
    k = np.tile(rng.standard_normal((1, 1, 8)), (2, 10, 1))
    ref = np.array([4 * sum(1.0 / (8 + i) for i in range(3) if t <= 7 + i) for t in range(10)])
    assert np.allclose(O.snapkv_votes(q, k), ref, rtol=1e-12)


@pytest.mark.parametrize("kernel", [1, 3, 7])
def test_pool_votes_matches_torch_pooling(kernel):
    """Max pooling = torch max_pool1d with -inf padding; average pooling = avg_pool1d with zero
    padding counted in the width (its default)."""
    rng = np.random.default_rng(kernel)
    v = rng.random(37)
    t = torch.from_numpy(v)[None, None]
    mx = torch.nn.functional.max_pool1d(t, kernel, stride=1, padding=kernel // 2)[0, 0].numpy()
    av = torch.nn.functional.avg_pool1d(t, kernel, stride=1, padding=kernel // 2)[0, 0].numpy()
    assert np.allclose(O.pool_votes(v, kernel, "max"), mx, rtol=0, atol=0)
    assert np.allclose(O.pool_votes(v, kernel, "avg"), av, rtol=1e-12, atol=1e-15)
