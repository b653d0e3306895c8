"""Plain, slow CPU oracle for the VeriCache draft-then-verify round.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module: only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline / reference leg call it. It shares no code
with the CUDA library (no helpers, tables, layouts code or constants generators).

Source: "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference" (technical summary
pages, in Japanese, French and German). The summary states the loop in its "Core algorithm"
section: (1) draft candidate tokens x with the compressed cache KV_comp, (2) verify all drafts
in one forward pass over the full cache KV_full, (3) accept up to the first mismatch, plus one
bonus token when every draft matches, then restart from the last accepted token. Its
"Architecture support" section names token-drop (SnapKV, KVzip) and quantisation (KIVI)
compressors behind one interface. Everything numeric (group sizes, bit widths, keep-set rules,
scale) is not on the pages; the readings used here are listed per function.

Precision: attention runs in float64 (softmax(q K^T / sqrt(d)) V, written out); quantisation
decisions run in IEEE float32 with round-to-nearest-even, because a float decides an integer
code there and both sides must take that decision in the same precision (the kernel's).

Every function here is pinned by tests/test_oracle_pins.py to closed forms, brute force on tiny
inputs and invariants; see that file for which pin guards which step.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

GROUP = 32  # quantisation group: 32 tokens per key channel, 32 channels per value token


# ----------------------------------------------------------------------------------------------
# a0. compression: token-drop keep-set
# ----------------------------------------------------------------------------------------------
def keep_set(importance: np.ndarray, keep: int, recent: int) -> np.ndarray:
    """Indices kept by token-drop compression, ascending int32.

    Reading (the pages name SnapKV/KVzip but define no scoring, "Architecture support"): the last
    `recent` tokens are always kept; the remaining keep-recent slots go to the tokens of
    [0, ctx-recent) with the largest importance, ties to the lower index; the union is returned
    sorted ascending. If keep >= ctx every token is kept.
    """
    imp = np.asarray(importance, dtype=np.float32)
    n = imp.shape[0]
    if keep >= n:
        return np.arange(n, dtype=np.int32)
    if not (0 <= recent <= keep):
        raise ValueError("need 0 <= recent <= keep")
    n_cand = n - recent
    cand = np.arange(n_cand)
    # sort by importance descending, then index ascending (lexsort: last key is primary)
    order = np.lexsort((cand, -imp[:n_cand].astype(np.float64)))
    top = order[: keep - recent]
    sel = np.concatenate([np.sort(top), np.arange(n_cand, n)])
    return sel.astype(np.int32)


# ----------------------------------------------------------------------------------------------
# a0. compression: groupwise asymmetric b-bit quantisation
# ----------------------------------------------------------------------------------------------
def fp16_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> float16, round to nearest even (IEEE conversion)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def quant_groups(x: np.ndarray, bits: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise each row of x (float32 [..., 32]) as one group.

    Reading (KIVI is named, not defined, on the pages): asymmetric min/max quantisation with
      s16 = fp16(fp32(max - min) / (2^b - 1)),  z16 = fp16(min),
      code = clamp(rint_half_even(fp32(x - f32(z16)) / f32(s16)), 0, 2^b - 1),  code = 0 if s16 == 0.
    Codes come from the stored fp16 scale and zero, so the codes and the dequantised values agree.
    Returns (codes uint8 [..., 32], s16 float16 [...], z16 float16 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    qmax = np.float32((1 << bits) - 1)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    s16 = fp16_rne((mx - mn) / qmax)
    z16 = fp16_rne(mn)
    s32 = s16.astype(np.float32)[..., None]
    z32 = z16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (x - z32) / s32
    codes = np.clip(np.rint(t), 0, qmax)
    codes = np.where(s32 == 0, 0, codes)
    return codes.astype(np.uint8), s16, z16


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack b-bit codes along the last axis, little-endian within a byte.

    Element e of a run lands in byte e // (8/b) at bit offset b * (e mod 8/b).
    """
    per = 8 // bits
    c = np.asarray(codes, dtype=np.uint8)
    n = c.shape[-1]
    assert n % per == 0
    c = c.reshape(c.shape[:-1] + (n // per, per)).astype(np.uint16)
    out = np.zeros(c.shape[:-1], dtype=np.uint16)
    for e in range(per):
        out |= c[..., e] << (bits * e)
    return out.astype(np.uint8)


def unpack(packed: np.ndarray, bits: int) -> np.ndarray:
    per = 8 // bits
    p = np.asarray(packed, dtype=np.uint8)
    mask = (1 << bits) - 1
    parts = [(p >> (bits * e)) & mask for e in range(per)]
    return np.stack(parts, axis=-1).reshape(p.shape[:-1] + (p.shape[-1] * per,)).astype(np.uint8)


def quant_layout(ctx: int, residual_min: int = 128) -> Tuple[int, int]:
    """(ng, n_res): quantised 32-token groups and bf16 residual rows.

    Reading: the configs keep "the last 128 tokens" in bf16; groups stay whole, so the first
    ng = floor((ctx - 128) / 32) groups are quantised and the residual is the remaining
    ctx - 32*ng tokens (128 to 159 of them).
    """
    ng = max(0, (ctx - residual_min) // GROUP)
    return ng, ctx - GROUP * ng


def frag_positions(d: int, kind: str) -> np.ndarray:
    """Storage order of the codes of one 32-token block (reading: the pages fix no format).

    The codes of a block are stored as 32-bit words w[half][j][lane] (half = 16-token half, j = one
    16-wide step over the channels, lane = 0..31). Word (half, j, lane) holds four pairs (i = 0..3)
    of (token, channel) positions, written out below; for keys the pairs run along channels, for
    values along tokens. Returns int [2][d/16][32][4][2][2]: (token, channel) of the low and the
    high code of pair i.
    """
    pos = np.zeros((2, d // 16, 32, 4, 2, 2), dtype=np.int64)
    for half in range(2):
        for j in range(d // 16):
            for lane in range(32):
                a, b = lane // 4, lane % 4
                if kind == "k":
                    t0, c0 = 16 * half + a, 16 * j + 2 * b
                    pairs = [((t0, c0), (t0, c0 + 1)), ((t0 + 8, c0), (t0 + 8, c0 + 1)),
                             ((t0, c0 + 8), (t0, c0 + 9)), ((t0 + 8, c0 + 8), (t0 + 8, c0 + 9))]
                else:
                    r0, k0 = 16 * j + a, 16 * half + 2 * b
                    pairs = [((k0, r0), (k0 + 1, r0)), ((k0, r0 + 8), (k0 + 1, r0 + 8)),
                             ((k0 + 8, r0), (k0 + 9, r0)), ((k0 + 8, r0 + 8), (k0 + 9, r0 + 8))]
                pos[half, j, lane] = np.array(pairs)
    return pos


def pack_block(codes: np.ndarray, bits: int, kind: str) -> np.ndarray:
    """Pack codes [..., 32 tokens, d] of whole blocks into their words, as little-endian bytes.

    4-bit: one word per (half, j, lane): pair i puts its low code at bits 4i and its high code at
    bits 16 + 4i. 2-bit: one word per (half, p, lane) covering steps j = 2p (pairs f = 0..3) and
    j = 2p + 1 (pairs f = 4..7): low code at bits 2f, high code at bits 16 + 2f.
    Output uint8 [..., 32 * d * bits / 8]: words in order [half][j or p][lane].
    """
    c = np.asarray(codes, dtype=np.uint32)
    d = c.shape[-1]
    lead = c.shape[:-2]
    pos = frag_positions(d, kind)
    if bits == 4:
        w = np.zeros(lead + (2, d // 16, 32), dtype=np.uint32)
        for i in range(4):
            sel = pos[:, :, :, i]                       # [2, d/16, 32, 2, 2]
            lo = c[..., sel[..., 0, 0], sel[..., 0, 1]]
            hi = c[..., sel[..., 1, 0], sel[..., 1, 1]]
            w |= (lo << np.uint32(4 * i)) | (hi << np.uint32(16 + 4 * i))
    else:
        w = np.zeros(lead + (2, d // 32, 32), dtype=np.uint32)
        for f in range(8):
            sel = pos[:, f // 4::2, :, f % 4]           # steps j = 2p + f // 4: [2, d/32, 32, 2, 2]
            lo = c[..., sel[..., 0, 0], sel[..., 0, 1]]
            hi = c[..., sel[..., 1, 0], sel[..., 1, 1]]
            w |= (lo << np.uint32(2 * f)) | (hi << np.uint32(16 + 2 * f))
    n_words = w.shape[-3] * w.shape[-2] * w.shape[-1]
    return np.ascontiguousarray(w.astype("<u4")).reshape(lead + (n_words,)).view(np.uint8)


def unpack_block(packed: np.ndarray, bits: int, kind: str, d: int) -> np.ndarray:
    """Inverse of pack_block: uint8 [..., 32 * d * bits / 8] -> codes uint8 [..., 32, d]."""
    p = np.ascontiguousarray(packed).view("<u4").astype(np.uint32)
    pos = frag_positions(d, kind)
    lead = p.shape[:-1]
    out = np.zeros(lead + (32, d), dtype=np.uint8)
    mask = np.uint32((1 << bits) - 1)
    if bits == 4:
        w = p.reshape(lead + (2, d // 16, 32))
        for i in range(4):
            lo = (w >> np.uint32(4 * i)) & mask
            hi = (w >> np.uint32(16 + 4 * i)) & mask
            out[..., pos[..., i, 0, 0], pos[..., i, 0, 1]] = lo
            out[..., pos[..., i, 1, 0], pos[..., i, 1, 1]] = hi
    else:
        w = p.reshape(lead + (2, d // 32, 32))
        for f in range(8):
            jj, i = f // 4, f % 4
            lo = (w >> np.uint32(2 * f)) & mask
            hi = (w >> np.uint32(16 + 2 * f)) & mask
            sel = pos[:, jj::2, :, i]  # steps j = 2p + jj
            out[..., sel[..., 0, 0], sel[..., 0, 1]] = lo
            out[..., sel[..., 1, 0], sel[..., 1, 1]] = hi
    return out


def quantize_kv(k: np.ndarray, v: np.ndarray, bits: int, residual_min: int = 128) -> dict:
    """Quantise one request's cache. k, v: float32 images of the bf16 cache, [Hkv][ctx][d].

    Keys: one group per (head, 32-token block, channel); values: one group per (head, token,
    32-channel group). Codes of each 32-token block are stored by pack_block (keys pair along
    channels, values along tokens). Layout (all C-contiguous):
      kc uint8 [Hkv][ng][32*d*b/8]   ks, kz float16 [Hkv][ng][d]
      vc uint8 [Hkv][ng][32*d*b/8]   vs, vz float16 [Hkv][Tq][d/32]
      k_res, v_res float32 [Hkv][n_res][d]  (tokens Tq..ctx-1, unchanged)
    """
    H, ctx, d = k.shape
    ng, n_res = quant_layout(ctx, residual_min)
    Tq = GROUP * ng
    kq = k[:, :Tq, :].reshape(H, ng, GROUP, d).transpose(0, 1, 3, 2)  # [H][ng][d][32 tokens]
    kcodes, ks, kz = quant_groups(kq, bits)
    vq = v[:, :Tq, :].reshape(H, Tq, d // GROUP, GROUP)               # [H][Tq][d/32][32 ch]
    vcodes, vs, vz = quant_groups(vq, bits)
    kblk = kcodes.transpose(0, 1, 3, 2)                                # [H][ng][32 tokens][d]
    vblk = vcodes.reshape(H, ng, GROUP, d)                             # [H][ng][32 tokens][d]
    return dict(bits=bits, ng=ng, n_res=n_res,
                kc=pack_block(kblk, bits, "k"), ks=ks, kz=kz,
                vc=pack_block(vblk, bits, "v"), vs=vs, vz=vz,
                k_res=k[:, Tq:, :].copy(), v_res=v[:, Tq:, :].copy())


def dequantize_kv(qkv: dict, d: int) -> Tuple[np.ndarray, np.ndarray]:
    """x_hat = code * f32(s16) + f32(z16) in float32, back in [Hkv][Tq][d] token-major order."""
    bits = qkv["bits"]
    kc = unpack_block(qkv["kc"], bits, "k", d).astype(np.float32)     # [H][ng][32][d]
    kh = kc * qkv["ks"].astype(np.float32)[:, :, None, :] + qkv["kz"].astype(np.float32)[:, :, None, :]
    H, ng = kh.shape[0], kh.shape[1]
    kh = kh.reshape(H, ng * GROUP, d)
    vc = unpack_block(qkv["vc"], bits, "v", d).astype(np.float32).reshape(H, ng * GROUP, d // GROUP, GROUP)
    vh = vc * qkv["vs"].astype(np.float32)[..., None] + qkv["vz"].astype(np.float32)[..., None]
    return kh.astype(np.float32), vh.reshape(H, ng * GROUP, d).astype(np.float32)


# ----------------------------------------------------------------------------------------------
# a1/a2. attention
# ----------------------------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible: np.ndarray | None = None) -> np.ndarray:
    """softmax(q k^T / sqrt(d)) v in float64 for one head.

    q [nq][d], k [n][d], v [n][d]; visible (bool [nq][n]) masks rows' keys, None = all visible.
    Reading: the pages print no attention formula; the scale 1/sqrt(d) is the standard one (also
    the one the position-independent-caching page on the same site writes in its score formula).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q @ k.T) / math.sqrt(q.shape[-1])
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    return (p @ v) / p.sum(axis=-1, keepdims=True)


def draft_attn(q: np.ndarray, k_main: np.ndarray, v_main: np.ndarray,
               k_win: np.ndarray, v_win: np.ndarray) -> np.ndarray:
    """One draft decode step of one request over the compressed cache ("Core algorithm", step 1).

    q [Hq][d]; KV_comp = the main rows k_main/v_main [Hkv][n][d] (kept rows of a token-drop cache,
    or the dequantised groups of a quantised cache) followed by the bf16 window k_win/v_win
    [Hkv][nw][d] (quantised residual, then the drafted tokens' own K/V up to and including the
    current one). GQA reading: query head h reads KV head h // (Hq / Hkv).
    Returns float64 [Hq][d].
    """
    Hq, d = q.shape
    Hkv = k_main.shape[0]
    G = Hq // Hkv
    out = np.empty((Hq, d), dtype=np.float64)
    for h in range(Hq):
        j = h // G
        K = np.concatenate([k_main[j], k_win[j]], axis=0)
        V = np.concatenate([v_main[j], v_win[j]], axis=0)
        out[h] = attention(q[h][None, :], K, V)[0]
    return out


def verify_attn(q: np.ndarray, k_full: np.ndarray, v_full: np.ndarray,
                k_new: np.ndarray, v_new: np.ndarray) -> np.ndarray:
    """Verification attention of one request ("Core algorithm", step 2): all n drafted tokens in one pass.

    q [n][Hq][d] are the queries at positions ctx..ctx+n-1; k_full/v_full [Hkv][ctx][d] is KV_full;
    k_new/v_new [Hkv][n][d] are the drafted tokens' K/V. Row i sees KV_full entirely and the new
    rows 0..i (causal among the drafts). GQA as in draft_attn. Returns float64 [n][Hq][d].
    """
    n, Hq, d = q.shape
    Hkv, ctx, _ = k_full.shape
    G = Hq // Hkv
    vis = np.ones((n, ctx + n), dtype=bool)
    vis[:, ctx:] = np.tril(np.ones((n, n), dtype=bool))
    out = np.empty((n, Hq, d), dtype=np.float64)
    for h in range(Hq):
        j = h // G
        K = np.concatenate([k_full[j], k_new[j]], axis=0)
        V = np.concatenate([v_full[j], v_new[j]], axis=0)
        out[:, h, :] = attention(q[:, h, :], K, V, vis)
    return out


# ----------------------------------------------------------------------------------------------
# a3. accept
# ----------------------------------------------------------------------------------------------
def accept(logits: np.ndarray, draft: Sequence[int], L: int) -> Tuple[List[int], int]:
    """Greedy accept of one request ("Core algorithm", step 3).

    logits [>= L+1][V]: row i is the full-cache prediction after the i-th verified input
    (row 0 follows the last accepted token, row i follows draft x_{i-1}); draft x_0..x_{L-1}.
    a_i = argmax of row i (first maximal index); n = first i < L with a_i != x_i, else L.
    Accepted tokens: x_0..x_{n-1} then a_n (the correction, or the bonus when n == L).
    Returns (tokens, n_acc = n + 1).
    """
    a = [int(np.argmax(logits[i])) for i in range(L + 1)]
    n = L
    for i in range(L):
        if a[i] != int(draft[i]):
            n = i
            break
    tokens = [int(draft[i]) for i in range(n)] + [a[n]]
    return tokens, n + 1


# ----------------------------------------------------------------------------------------------
# a0 input. SnapKV-style importance (observation-window votes, pooled)
# ----------------------------------------------------------------------------------------------
def snapkv_votes(q_obs: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Votes of the observation window ("Architecture support" names SnapKV among the token-drop
    compressors; the pages do not define its scoring, this is the plain reading).

    q_obs [W][Hq][d]: queries of the last W context tokens (window query i at position
    ctx - W + i); k [Hkv][ctx][d]: KV_full keys. Query head h reads KV head h // (Hq/Hkv). Row
    (i, h) takes the softmax of q k^T / sqrt(d) over keys 0 .. ctx - W + i; vote[t] is the sum of
    key t's weights over every row. float64, returns [ctx]."""
    W, Hq, d = q_obs.shape
    Hkv, ctx, _ = k.shape
    G = Hq // Hkv
    votes = np.zeros(ctx, dtype=np.float64)
    for h in range(Hq):
        scores = q_obs[:, h, :].astype(np.float64) @ k[h // G].astype(np.float64).T / math.sqrt(d)
        for i in range(W):
            pos = ctx - W + i
            s = scores[i, : pos + 1]
            a = np.exp(s - s.max())
            votes[: pos + 1] += a / a.sum()
    return votes


def pool_votes(votes: np.ndarray, kernel: int, kind: str) -> np.ndarray:
    """1-D pooling of width `kernel` (odd) centred on each token: "max" takes the largest vote in
    range, "avg" the in-range sum divided by the width (zero padding outside the context)."""
    half = kernel // 2
    n = len(votes)
    out = np.empty(n, dtype=np.float64)
    for t in range(n):
        win = votes[max(0, t - half): min(n, t + half + 1)]
        out[t] = win.max() if kind == "max" else win.sum() / kernel
    return out


def snapkv_importance(q_obs: np.ndarray, k: np.ndarray, pool_kernel: int = 7, pool: str = "max") -> np.ndarray:
    return pool_votes(snapkv_votes(q_obs, k), pool_kernel, pool)


# ----------------------------------------------------------------------------------------------
# staggering plan (two alternating groups)
# ----------------------------------------------------------------------------------------------
def stagger_period2(costs: Sequence[Tuple[int, int, int]], groups: Sequence[int]) -> int:
    """Twice the steady-state period of the two-group stagger ("Cross-resource staggering (P1)";
    the pages fix no schedule, this is the reading stated with the library's planner).

    costs[r] = (d, v, s): draft-phase time, verification-and-accept time and host-link copy time of
    request r (s = 0 when its KV_full stays in HBM); groups[r] in {0, 1}. Schedule: the compute
    stream repeats [draft 0, verify 1, draft 1, verify 0], the copy stream [copy 1, copy 0]; a
    verification waits for its group's copy of the same period, a copy for its group's previous
    verification. The period is the largest cycle mean of that max-plus system:
        T = max(D + V, S, S_0 + V_0, S_1 + V_1, (S + V + D_0) / 2, (S + V + D_1) / 2).
    """
    D = [0, 0]
    S = [0, 0]
    V = [0, 0]
    for (d, v, s), g in zip(costs, groups):
        D[g] += d
        S[g] += s
        V[g] += v
    Dt, St, Vt = sum(D), sum(S), sum(V)
    return max(2 * (Dt + Vt), 2 * St, 2 * (S[0] + V[0]), 2 * (S[1] + V[1]), St + Vt + D[0], St + Vt + D[1])


def stagger_period(costs: Sequence[Tuple[int, int, int]], groups: Sequence[int]) -> int:
    """The period, rounded up to a whole unit."""
    return (stagger_period2(costs, groups) + 1) // 2


def stagger_phase_work(costs: Sequence[Tuple[int, int, int]], groups: Sequence[int]) -> int:
    """The longer phase's GPU work of a split: phase 1 drafts group 0 and verifies group 1, phase 2
    the reverse, so max(D_0 + V_1, D_1 + V_0). Splits of equal period are told apart by it (the
    balanced one leaves each phase enough drafting to cover the other group's copy)."""
    D = [0, 0]
    V = [0, 0]
    for (d, v, s), g in zip(costs, groups):
        D[g] += d
        V[g] += v
    return max(D[0] + V[1], D[1] + V[0])


def plan_stagger(costs: Sequence[Tuple[int, int, int]]) -> Tuple[List[int], int]:
    """Best split by brute force: every assignment with request 0 in group 0 and, for n >= 2, at
    least one request in group 1; minimum period (compared as 2T), then minimum phase work
    (stagger_phase_work), then the smallest sum of groups[r] * 2^(r-1). Returns (groups, period)."""
    import itertools
    n = len(costs)
    best = None
    for tail in itertools.product((0, 1), repeat=n - 1):
        if n >= 2 and not any(tail):
            continue
        groups = [0] + list(tail)
        key = sum(g << (r - 1) for r, g in enumerate(groups) if r >= 1)
        t2 = stagger_period2(costs, groups)
        ph = stagger_phase_work(costs, groups)
        if best is None or (t2, ph, key) < best[:3]:
            best = (t2, ph, key, groups)
    return best[3], (best[0] + 1) // 2


# ----------------------------------------------------------------------------------------------
# helpers for whole requests
# ----------------------------------------------------------------------------------------------
def bf16_to_f32(t) -> np.ndarray:
    """float32 image of a bf16 torch tensor (exact)."""
    import torch
    return t.detach().to("cpu").to(torch.float32).numpy()


def comp_main_rows(mode: str, k: np.ndarray, v: np.ndarray, *, idx=None, qkv=None):
    """KV_comp main rows as float32 [Hkv][n][d] for draft_attn."""
    if mode == "drop":
        return k[:, idx, :], v[:, idx, :]
    kh, vh = dequantize_kv(qkv, k.shape[2])
    return kh, vh


def draft_round(q: np.ndarray, k_main, v_main, k_win0, v_win0, k_new, v_new) -> np.ndarray:
    """All L draft steps of one request: step s attends main + window0 + new[0..s]. Returns [L][Hq][d]."""
    L = q.shape[0]
    out = np.empty(q.shape, dtype=np.float64)
    for s in range(L):
        kw = np.concatenate([k_win0, k_new[: s + 1].transpose(1, 0, 2)], axis=1)
        vw = np.concatenate([v_win0, v_new[: s + 1].transpose(1, 0, 2)], axis=1)
        out[s] = draft_attn(q[s], k_main, v_main, kw, vw)
    return out
