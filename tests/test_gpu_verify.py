"""GPU parity of verification attention (tcgen05/TMEM kernel) against the oracle.

Row i of a request attends to KV_full[0:ctx] and to drafted rows 0..i. Cases span several KV tiles
with a ragged last tile, 1 to 3 query-row tiles (G * n_rows = 32 ... 320), units split across CTAs
and whole units, d = 64 and 128; full sizes are sampled per (request, KV head)."""
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


def _fill_window(bt):
    for r in bt.reqs:
        r.k_win[:, r.n_res: r.n_res + r.L].copy_(r.k_new.transpose(0, 1))
        r.v_win[:, r.n_res: r.n_res + r.L].copy_(r.v_new.transpose(0, 1))


def _check(w, reqs, heads=None, env_ctas=None, monkeypatch=None):
    if env_ctas is not None:
        monkeypatch.setenv("VC_VERIFY_CTAS", str(env_ctas))
    bt = make_batch(w, reqs)
    _fill_window(bt)
    bt.verify()
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    G = w.Hq // w.Hkv
    for i, b in enumerate(reqs):
        r = bt.reqs[i]
        q, kf, vf = f32(r.q), f32(r.k_full), f32(r.v_full)
        kn, vn = f32(r.k_new).transpose(1, 0, 2), f32(r.v_new).transpose(1, 0, 2)
        hs = range(w.Hkv) if heads is None else heads
        for hk in hs:
            sel = slice(hk * G, (hk + 1) * G)
            ref = O.verify_attn(q[:, sel], kf[hk:hk + 1], vf[hk:hk + 1], kn[hk:hk + 1], vn[hk:hk + 1])
            assert_attn_close(r.o_verify[:, sel], ref, f"{w.name} b{b} hk{hk}")


def test_verify_tiny():
    _check(configs.tiny(), [0])


def test_verify_llama8b_scaled():
    _check(configs.scaled(configs.llama8b_drop(), ctx_div=16, batch=3), [0, 1, 2])


def test_verify_qwen_ragged_rows():
    """125 query rows per KV head (L 25 x G 5), context not a multiple of 64."""
    w = configs.scaled(configs.qwen32b_quant2(), ctx_div=64, batch=2)
    w.ctx = [1000, 1087]
    _check(w, [0, 1])


def test_verify_llama70b_three_row_tiles():
    """320 query rows per KV head (L 40 x G 8): three 128-row tiles."""
    _check(configs.scaled(configs.llama70b_offload4(), ctx_div=128, batch=2), [0, 1])


def test_verify_mixed_ragged():
    w = configs.scaled(configs.mixed_serving(), ctx_div=64, batch=6)
    _check(w, list(range(6)))


@pytest.mark.parametrize("ctas", [1, 3, 7, 1000])
def test_verify_split_layouts(ctas, monkeypatch):
    """The same inputs cut into 1 CTA (no splits), a few CTAs, and one CTA per tile."""
    w = configs.scaled(configs.llama8b_drop(), ctx_div=64, batch=2, L=9)
    _check(w, [0, 1], env_ctas=ctas, monkeypatch=monkeypatch)


def _mode_env(monkeypatch, mode):
    """rows: every row tile of a head in one CTA (VC_VERIFY_ROWS=1); default: two-tile heads in pair
    mode and the rest one unit per row tile (a launch per kind); trio: the default plus three-tile
    heads in trio mode (VC_VERIFY_TRIO=1); units: one unit per row tile for every head
    (VC_VERIFY_PAIR=0)."""
    monkeypatch.setenv("VC_VERIFY_ROWS", "1" if mode == "rows" else "0")
    monkeypatch.setenv("VC_VERIFY_PAIR", "0" if mode == "units" else "1")
    if mode == "trio":
        monkeypatch.setenv("VC_VERIFY_TRIO", "1")
    else:
        monkeypatch.delenv("VC_VERIFY_TRIO", raising=False)


@pytest.mark.parametrize("ctas", [1, 5, 1000])
@pytest.mark.parametrize("mode", ["rows", "trio", "default"])
def test_verify_row_tiles_split_layouts(ctas, mode, monkeypatch):
    """More than 128 query rows per KV head (L 40 x G 8 = 320: three row tiles), ragged context:
    every row tile of a KV head in one CTA with one softmax warpgroup (row-tile mode), in trio mode
    (two softmax warpgroups, tiles 0 and 2 on the first) and one unit per row tile (the default),
    each cut into one CTA, a few CTAs and one CTA per KV tile, so heads split across CTAs merge
    their partials."""
    _mode_env(monkeypatch, mode)
    w = configs.scaled(configs.llama70b_offload4(), ctx_div=256, batch=2)
    w.ctx = [517, 1000]
    _check(w, [0, 1], env_ctas=ctas, monkeypatch=monkeypatch)


@pytest.mark.parametrize("mode", ["trio", "default", "units"])
@pytest.mark.parametrize("d128", [True, False])
def test_verify_one_to_four_row_tiles(mode, d128, monkeypatch):
    """One call whose KV heads have one row tile (L 25 x G 4 = 100 rows), two (160), three (280 and
    384, the most trio mode takes) and four (388): with trio mode on, a launch each for the heads
    of one, three or four tiles (a unit per tile), the pair-mode heads and the trio-mode heads. d =
    128 and d = 64 (the tiny shape), both with G 4."""
    _mode_env(monkeypatch, mode)
    if d128:
        w = configs.scaled(configs.mixed_serving(), ctx_div=64, batch=5)
    else:
        w = configs.scaled(configs.tiny(), batch=5)
        w.ctx = [300, 1000, 517, 260, 2000]
    w.L = [25, 40, 70, 96, 97]
    _check(w, list(range(5)))


@pytest.mark.parametrize("mode", ["rows", "default", "units"])
def test_verify_row_tiles_mixed_one_and_two(mode, monkeypatch):
    """One call with KV heads of one row tile (L 25 x G 4 = 100 rows, L 32: 128) and of two (L 40:
    160 rows, L 33: 132): the row-tile mode holds both kinds of units; by default the two-tile
    requests go to a pair-mode launch and the others to the one-unit-per-tile launch."""
    _mode_env(monkeypatch, mode)
    w = configs.scaled(configs.mixed_serving(), ctx_div=32, batch=4)
    w.L = [25, 40, 33, 32]
    _check(w, [0, 1, 2, 3])


@pytest.mark.parametrize("ctas", [1, 5, 1000])
@pytest.mark.parametrize("mode", ["default", "units"])
def test_verify_two_row_tiles_split_layouts(ctas, mode, monkeypatch):
    """Two row tiles per KV head (L 20 x G 8 = 160 rows), ragged contexts, the pair mode's launch
    cut into one CTA, a few and one CTA per KV tile: the two warpgroups' partials of split heads
    merge through the combine kernel."""
    _mode_env(monkeypatch, mode)
    w = configs.scaled(configs.llama70b_offload4(), ctx_div=256, batch=3, L=20)
    w.ctx = [517, 1000, 64]
    _check(w, [0, 1, 2], env_ctas=ctas, monkeypatch=monkeypatch)


@pytest.mark.parametrize("L,ctx", [(1, 1), (1, 64), (70, 65), (64, 200), (3, 5000)])
def test_verify_edges(L, ctx):
    """One drafted row, one context token, drafts spanning two tiles, exact tile multiples."""
    w = configs.scaled(configs.tiny(), batch=1, L=L)
    w.ctx = [ctx]
    _check(w, [0])


def test_verify_llama8b_full_size_sampled():
    w = configs.llama8b_drop()
    _check(w, list(range(8)), heads=[0, 5])


def test_verify_qwen32b_full_size_sampled():
    w = configs.qwen32b_quant2()
    _check(w, list(range(16)), heads=[2])


@pytest.mark.parametrize("ranges", [[(0, 8)], [(0, 3), (3, 5), (5, 8)], [(h, h + 1) for h in range(8)], [(2, 6)]])
def test_verify_head_ranges(ranges):
    """vc_verify_attn_heads over KV-head ranges: the heads in the ranges match the oracle and the
    other heads' outputs are left as they were (NaN here)."""
    import lossless_compressed_kv_vc_gb300 as vc
    w = configs.scaled(configs.llama8b_drop(), ctx_div=32, batch=3, L=7)
    bt = make_batch(w, [0, 1, 2])
    _fill_window(bt)
    for r in bt.reqs:
        r.o_verify.fill_(float("nan"))
    arr = bt.verify_requests()
    for h0, h1 in ranges:
        vc.vc_verify_attn_heads(bt.shape, arr, h0, h1, bt.ws_verify, bt.dev_status)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    G = w.Hq // w.Hkv
    done = set(h for h0, h1 in ranges for h in range(h0, h1))
    for i, r in enumerate(bt.reqs):
        q, kf, vf = f32(r.q), f32(r.k_full), f32(r.v_full)
        kn, vn = f32(r.k_new).transpose(1, 0, 2), f32(r.v_new).transpose(1, 0, 2)
        for hk in range(w.Hkv):
            sel = slice(hk * G, (hk + 1) * G)
            if hk in done:
                ref = O.verify_attn(q[:, sel], kf[hk:hk + 1], vf[hk:hk + 1], kn[hk:hk + 1], vn[hk:hk + 1])
                assert_attn_close(r.o_verify[:, sel], ref, f"b{i} hk{hk}")
            else:
                assert torch.isnan(r.o_verify[:, sel].float()).all(), f"b{i} hk{hk} written outside the range"


def test_verify_head_range_validation():
    import lossless_compressed_kv_vc_gb300 as vc
    w = configs.tiny()
    bt = make_batch(w, [0])
    arr = bt.verify_requests()
    for h0, h1 in [(-1, 1), (1, 1), (0, w.Hkv + 1), (2, 1)]:
        st = vc.vc_verify_attn_heads(bt.shape, arr, h0, h1, bt.ws_verify, bt.dev_status, raise_on_error=False)
        assert st == vc.VC_ERR_INVALID
