"""The C-ABI library builds for sm_103a, loads, and exports every entry point include/vc.h declares.
No compute calls: these run without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import LIB_PATH
    return ctypes.CDLL(LIB_PATH)


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(vc_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_round_calls():
    names = declared_symbols()
    for n in ["vc_compress_kv", "vc_draft_attn", "vc_verify_attn", "vc_verify_attn_heads", "vc_accept", "vc_stage_full_kv", "vc_append_kv", "vc_snapkv_importance", "vc_plan_stagger",
              "vc_workspace_size", "vc_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.vc_status_string.restype = ctypes.c_char_p
    assert lib.vc_status_string(0) == b"ok"
    assert b"page-locked" in lib.vc_status_string(4)
    assert lib.vc_version() >= 100


def test_binding_names_match_header():
    import lossless_compressed_kv_vc_gb300 as vc
    for n in declared_symbols():
        assert hasattr(vc, n), n


def test_validation_rejects_without_launching(lib):
    """Host-side validation runs before any CUDA call, so it is testable without a GPU."""
    import lossless_compressed_kv_vc_gb300 as vc
    bad = vc.vc_shape(0, 8, 2, 64)
    assert vc.vc_draft_attn(bad, None, stream=0, raise_on_error=False) == vc.VC_ERR_INVALID
    shp = vc.vc_shape(1, 8, 2, 96)
    assert vc.vc_verify_attn(shp, None, stream=0, raise_on_error=False) in (vc.VC_ERR_INVALID, vc.VC_ERR_UNSUPPORTED)
    assert vc.vc_accept(0, 4, 10, 16, 16, 16, 16, 16, stream=0, raise_on_error=False) == vc.VC_ERR_INVALID
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, bad) == 0
    ok = vc.vc_shape(8, 32, 8, 128)
    assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, ok) > 0


def test_draft_counter_block_does_not_depend_on_the_shape(lib):
    """The draft workspace starts with a fixed block of arrival counters (VC_DRAFT_COUNTER_BYTES,
    room for VC_DRAFT_MAX_KV_HEADS heads), so a workspace zero-filled once keeps zero counters for
    calls of any shape: the partials start at the same offset whatever Hkv is, and a workspace's
    size grows with the partials only."""
    import lossless_compressed_kv_vc_gb300 as vc
    hdr = open(os.path.join(ROOT, "include", "vc.h")).read()
    assert re.search(r"#define VC_DRAFT_MAX_KV_HEADS\s+%d\b" % vc.VC_DRAFT_MAX_KV_HEADS, hdr)
    assert re.search(r"#define VC_DRAFT_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)32 << 20\)", hdr)
    assert vc.VC_DRAFT_COUNTER_BYTES == vc.VC_DRAFT_MAX_KV_HEADS * vc.VC_MAX_BATCH * 4
    for B, Hq, Hkv, d in ((1, 8, 2, 64), (8, 32, 8, 128), (16, 40, 8, 128), (4, 256, 256, 128)):
        ws = vc.vc_workspace_size(vc.VC_CALL_DRAFT, vc.vc_shape(B, Hq, Hkv, d))
        assert ws > vc.VC_DRAFT_COUNTER_BYTES
    # beyond the counter block's heads: refused before anything is launched
    big = vc.vc_shape(1, 257, 257, 128)
    req = (vc.vc_draft_req * 1)()
    assert vc.vc_draft_attn(big, req, stream=0, raise_on_error=False) == vc.VC_ERR_UNSUPPORTED


def test_draft_workspace_covers_the_widest_wave(lib):
    """The draft workspace holds, per KV head, a partial slot for every CTA of the widest draft
    launch of any cache kind (one wave: 4 CTAs per SM for quantised caches with G <= 8, 3 for
    token drop; 152 SMs when no GPU answers) plus two per request, each G (d + 1) floats, after the
    fixed counter block. Sizing by one kind alone undersizes it as soon as the kinds' waves
    differ."""
    import lossless_compressed_kv_vc_gb300 as vc
    sms, widest = 152, 4
    for B, Hq, Hkv, d in ((1, 8, 2, 64), (8, 32, 8, 128), (16, 40, 8, 128), (32, 32, 8, 128), (2, 64, 8, 128)):
        G = Hq // Hkv
        per_head = max(1, widest * sms // Hkv)
        need = vc.VC_DRAFT_COUNTER_BYTES + Hkv * (per_head + 2 * B) * G * (d + 1) * 4
        assert vc.vc_workspace_size(vc.VC_CALL_DRAFT, vc.vc_shape(B, Hq, Hkv, d)) >= need, (B, Hq, Hkv, d)


def test_comp_bytes_follows_the_layout_rule():
    """vc_comp_bytes (host only) against the oracle's statement of the quantised layout: blocks and
    residual at ctx, block capacity for the grown context, window rows = the largest residual on the
    way there + drafts + 1, and each buffer's bytes from its documented shape."""
    import oracle as O
    import lossless_compressed_kv_vc_gb300 as vc
    sh = vc.vc_shape(1, 32, 8, 128)
    for ctx, grow, bits, L in ((1000, 0, 2, 8), (65536, 0, 2, 25), (131072, 0, 4, 40), (100, 0, 2, 3),
                               (300, 2, 4, 5), (300, 200, 2, 5), (128, 40, 2, 1), (160, 0, 4, 0)):
        sz = vc.vc_comp_bytes(sh, vc.VC_QUANT, bits, ctx, ctx + grow, 0, 128, L)
        ng, nr = O.quant_layout(ctx, 128)
        cap = max(O.quant_layout(ctx + grow, 128)[0], 1)
        res_max = max([O.quant_layout(c, 128)[1] for c in range(ctx, ctx + grow + 1)])
        assert (sz.ng, sz.n_res, sz.ng_cap) == (ng, nr, cap)
        assert res_max <= sz.win_cap - L - 1 <= max(nr, 128 + 31)  # covers every residual on the way
        assert sz.codes_bytes == 8 * cap * 32 * 128 * bits // 8
        assert sz.kscale_bytes == 8 * cap * 128 * 2 and sz.vscale_bytes == 8 * 32 * cap * 4 * 2
        assert sz.win_bytes == 8 * sz.win_cap * 128 * 2
    sz = vc.vc_comp_bytes(sh, vc.VC_TOKEN_DROP, 0, 32768, 32768, 8192, 128, 32)
    assert (sz.keep, sz.idx_bytes, sz.rows_bytes, sz.win_cap) == (8192, 8192 * 4, 8 * 8192 * 128 * 2, 33)
    assert vc.vc_comp_bytes(sh, vc.VC_TOKEN_DROP, 0, 100, 100, 500).keep == 100
    for args in ((vc.VC_QUANT, 3, 1000), (vc.VC_QUANT, 2, 0), (7, 2, 1000)):
        with pytest.raises(vc.VCError):
            vc.vc_comp_bytes(sh, *args)


def test_append_validation_rejects_without_launching(lib):
    """vc_append_kv checks capacities before launching; a call with nothing to append launches
    nothing and succeeds. The pointers are fake (aligned, never dereferenced on these paths)."""
    import lossless_compressed_kv_vc_gb300 as vc
    shp = vc.vc_shape(1, 8, 2, 64)

    def call(ctx, cap, n, quant=False, ng=0, ng_cap=0, bits=2, win_cap=512):
        full = (vc.vc_kv_full * 1)()
        full[0].k, full[0].v, full[0].ctx, full[0].cap = 1 << 12, 1 << 13, ctx, cap
        comp = (vc.vc_kv_comp * 1)()
        c = comp[0]
        c.mode, c.bits, c.ng, c.ng_cap, c.win_cap, c.n_win = (vc.VC_QUANT if quant else vc.VC_TOKEN_DROP), bits, ng, \
            ng_cap, win_cap, 0
        for f in ("kc", "ks", "kz", "vc", "vs", "vz", "k_win", "v_win", "idx"):
            setattr(c, f, 1 << 14)
        req = (vc.vc_append_req * 1)()
        req[0].k_rows, req[0].v_rows, req[0].n_rows = 1 << 15, 1 << 16, n
        st = vc.vc_append_kv(shp, full, comp, req, 128, None, stream=0, raise_on_error=False)
        return st, full[0].ctx
    assert call(100, 110, 11) == (vc.VC_ERR_INVALID, 100)                 # past KV_full's capacity
    assert call(100, 110, -1)[0] == vc.VC_ERR_INVALID
    assert call(100, 110, 0) == (vc.VC_OK, 100)                           # nothing to do
    assert call(300, 1000, 0, quant=True, ng=5, ng_cap=5) == (vc.VC_OK, 300)
    assert call(300, 1000, 32, quant=True, ng=5, ng_cap=5)[0] == vc.VC_ERR_INVALID   # needs block 6
    assert call(300, 1000, 117, quant=True, ng=5, ng_cap=50)[0] == vc.VC_ERR_UNSUPPORTED  # 140+117 rows
    assert call(300, 1000, 8, quant=True, ng=5, ng_cap=50, bits=3)[0] == vc.VC_ERR_UNSUPPORTED
    assert call(300, 1000, 8, quant=True, ng=5, ng_cap=50, win_cap=100)[0] == vc.VC_ERR_INVALID  # residual > window


def test_verify_head_range_rejected_before_launch(lib):
    import lossless_compressed_kv_vc_gb300 as vc
    shp = vc.vc_shape(1, 8, 2, 64)
    arr = (vc.vc_verify_req * 1)()
    for h0, h1 in [(-1, 1), (1, 1), (0, 3), (2, 1)]:
        assert vc.vc_verify_attn_heads(shp, arr, h0, h1, None, None, stream=0, raise_on_error=False) == vc.VC_ERR_INVALID


@pytest.mark.parametrize("env,rows,expect", [
    ({}, [32], 2),                               # one row tile (G 4: 128 rows): units
    ({}, [25, 40], 4),                           # one and two tiles: units + pair mode
    ({"VC_VERIFY_PAIR": "0"}, [25, 40], 2),      # pair mode off: units only
    ({}, [25, 40, 70, 97], 4),                   # three and four tiles go to units by default
    ({"VC_VERIFY_TRIO": "1"}, [25, 40, 70], 6),  # units + pair + trio
    ({"VC_VERIFY_TRIO": "1"}, [70, 96], 2),      # trio only (280 and 384 rows)
    ({"VC_VERIFY_ROWS": "1"}, [25, 40, 70], 2),  # row-tile mode over the whole call
    ({"VC_VERIFY_ROWS": "1"}, [25, 97], 2),      # four tiles: no row-tile mode; one and four: units
])
def test_verify_launch_count(lib, monkeypatch, env, rows, expect):
    """vc_verify_launches: two kernels (verification and merge) per kind of launch the requests
    need, host only (the pointers are never dereferenced)."""
    import lossless_compressed_kv_vc_gb300 as vc
    for k in ("VC_VERIFY_PAIR", "VC_VERIFY_TRIO", "VC_VERIFY_ROWS"):
        monkeypatch.delenv(k, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    shp = vc.vc_shape(len(rows), 32, 8, 128)                     # G 4
    arr = (vc.vc_verify_req * len(rows))()
    for b, n in enumerate(rows):
        e = arr[b]
        e.full.k, e.full.v, e.full.ctx, e.full.cap = 1 << 12, 1 << 13, 1000, 1000
        e.q, e.k_new, e.v_new, e.o = 1 << 14, 1 << 15, 1 << 16, 1 << 17
        e.new_cap, e.n_rows = n, n
    assert vc.vc_verify_launches(shp, arr) == expect
    arr[0].n_rows = 0                                             # refused by vc_verify_attn too
    assert vc.vc_verify_launches(shp, arr) == -1


def test_plan_stagger_equals_oracle_brute_force():
    """The library's Gray-code enumeration against the oracle's itertools brute force: the same
    split (with the same tie-break) and period on random integer costs, resident requests mixed in."""
    import numpy as np
    import oracle as O
    import lossless_compressed_kv_vc_gb300 as vc
    rng = np.random.default_rng(11)
    for n in list(range(1, 13)) + [12, 12]:
        for _ in range(6):
            costs = []
            for r in range(n):
                d, v, s = (int(x) for x in rng.integers(0, 5_000_000, 3))
                if rng.random() < 0.4:
                    s = 0
                costs.append((d, v, s))
            st, groups, t = vc.vc_plan_stagger(costs)
            ref_groups, ref_t = O.plan_stagger(costs)
            assert st == vc.VC_OK and groups == ref_groups and t == ref_t, (n, costs)
            assert vc.vc_stagger_period(costs, groups)[1] == O.stagger_period(costs, groups)


def test_plan_stagger_ties_and_limits():
    import time
    import lossless_compressed_kv_vc_gb300 as vc
    st, groups, t = vc.vc_plan_stagger([(0, 10, 10)] * 4)
    assert groups == [0, 1, 1, 0] and t == 40
    costs = [(1000 + 37 * r, 100, 900 + 53 * r) for r in range(vc.VC_STAGGER_MAX)]
    t0 = time.time()
    st, groups, t = vc.vc_plan_stagger(costs)
    assert st == vc.VC_OK and time.time() - t0 < 5.0
    assert vc.vc_stagger_period(costs, groups)[1] == t
    assert vc.vc_plan_stagger(costs + [(1, 1, 1)], raise_on_error=False)[0] == vc.VC_ERR_UNSUPPORTED
    assert vc.vc_plan_stagger([(1, -1, 0)], raise_on_error=False)[0] == vc.VC_ERR_INVALID
    assert vc.vc_plan_stagger([(1 << 41, 0, 0)], raise_on_error=False)[0] == vc.VC_ERR_INVALID
    assert vc.vc_stagger_period([(1, 1, 1)], [2], raise_on_error=False)[0] == vc.VC_ERR_INVALID


def _random_costs(rng, n):
    costs = []
    for _ in range(n):
        d, v, s = (int(x) for x in rng.integers(0, 5_000_000, 3))
        if rng.random() < 0.4:
            s = 0  # KV_full resident in HBM
        costs.append((d, v, s))
    return costs


def test_plan_stagger_local_is_a_local_optimum_of_the_oracle_period():
    """Beyond the exact planner: the split is valid, its period is the oracle's period of that
    split, and no single move or swap of two requests lowers the oracle's 2T."""
    import numpy as np
    import oracle as O
    import lossless_compressed_kv_vc_gb300 as vc
    rng = np.random.default_rng(23)
    for n in (2, 3, 5, 9, 17, 25, 33, 64):
        for _ in range(3):
            costs = _random_costs(rng, n)
            st, groups, t = vc.vc_plan_stagger_local(costs)
            assert st == vc.VC_OK and groups[0] == 0 and 0 < sum(groups) < n
            assert t == O.stagger_period(costs, groups)
            t2 = O.stagger_period2(costs, groups)
            for r in range(n):
                g = list(groups)
                g[r] ^= 1
                if 0 < sum(g) < n:
                    assert O.stagger_period2(costs, g) >= t2, (n, r)
            for r in [i for i in range(n) if groups[i] == 0]:
                for q in [i for i in range(n) if groups[i] == 1]:
                    g = list(groups)
                    g[r], g[q] = 1, 0
                    assert O.stagger_period2(costs, g) >= t2, (n, r, q)


def test_plan_stagger_local_against_the_exact_split():
    """Never below the oracle's exact optimum (it cannot be), and on these random batches it finds it."""
    import numpy as np
    import oracle as O
    import lossless_compressed_kv_vc_gb300 as vc
    rng = np.random.default_rng(29)
    found = total = 0
    for n in range(2, 12):
        for _ in range(8):
            costs = _random_costs(rng, n)
            t = vc.vc_plan_stagger_local(costs)[2]
            t_exact = O.plan_stagger(costs)[1]
            assert t >= t_exact
            found += t == t_exact
            total += 1
    assert found >= 0.9 * total, (found, total)


def test_plan_stagger_local_limits_and_engine_choice():
    import time
    import numpy as np
    import oracle as O
    import lossless_compressed_kv_vc_gb300 as vc
    from lossless_compressed_kv_vc_gb300 import engine
    st, groups, t = vc.vc_plan_stagger_local([(5, 3, 7)])
    assert (st, groups, t) == (vc.VC_OK, [0], O.stagger_period([(5, 3, 7)], [0]))
    rng = np.random.default_rng(31)
    big = _random_costs(rng, vc.VC_STAGGER_LOCAL_MAX)
    t0 = time.time()
    st, groups, t = vc.vc_plan_stagger_local(big)
    assert st == vc.VC_OK and time.time() - t0 < 10.0 and 0 < sum(groups) < len(big)
    assert vc.vc_stagger_period(big, groups)[1] == t
    assert vc.vc_plan_stagger_local(big + [(1, 1, 1)], raise_on_error=False)[0] == vc.VC_ERR_UNSUPPORTED
    assert vc.vc_plan_stagger_local([], raise_on_error=False)[0] == vc.VC_ERR_INVALID
    assert vc.vc_plan_stagger_local([(1, -1, 0)], raise_on_error=False)[0] == vc.VC_ERR_INVALID
    # the engine plans exactly up to VC_STAGGER_MAX requests and by local search beyond
    small = _random_costs(rng, 10)
    a, b, t = engine.plan_groups(small)
    assert t == O.plan_stagger(small)[1] and sorted(a + b) == list(range(10))
    many = _random_costs(rng, vc.VC_STAGGER_MAX + 6)
    a, b, t = engine.plan_groups(many)
    assert a and b and sorted(a + b) == list(range(len(many)))
    assert t == vc.vc_plan_stagger_local(many)[2]


def test_importance_validation_rejects_without_launching(lib):
    import lossless_compressed_kv_vc_gb300 as vc
    arr = (vc.vc_importance_req * 1)()
    arr[0].full.k, arr[0].full.v, arr[0].full.ctx, arr[0].full.cap = 1 << 12, 1 << 13, 100, 100
    arr[0].q_obs, arr[0].importance = 1 << 14, 1 << 15
    shp = vc.vc_shape(1, 8, 2, 128)  # G = 4
    call = lambda W, k=7, kind=vc.VC_POOL_MAX, s=shp: vc.vc_snapkv_importance(s, arr, W, k, kind, None, None,
                                                                                stream=0, raise_on_error=False)
    assert call(6) == vc.VC_ERR_WORKSPACE         # 24 window rows: any count is fine
    assert call(8, k=4) == vc.VC_ERR_INVALID      # even pooling width
    assert call(8, k=67) == vc.VC_ERR_UNSUPPORTED  # wider than 65
    assert call(8, kind=2) == vc.VC_ERR_INVALID
    assert call(8) == vc.VC_ERR_WORKSPACE         # valid request, no workspace
    assert call(8, s=vc.vc_shape(1, 8, 2, 96)) == vc.VC_ERR_UNSUPPORTED
    arr[0].full.ctx = 7
    assert call(8) == vc.VC_ERR_INVALID           # context shorter than the window
    assert vc.vc_importance_workspace_size(shp, 8, 100) > 0


def test_binding_refuses_to_import_without_the_library(tmp_path):
    """No fallback path: the package raises ImportError when libvc.so is absent."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "lossless_compressed_kv_vc_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "lossless_compressed_kv_vc_gb300", "__init__.py"), pkg / "__init__.py")
    code = ("import sys; sys.path.insert(0, %r)\n"
            "try:\n    import lossless_compressed_kv_vc_gb300\nexcept ImportError as e:\n"
            "    print('refused:', e); sys.exit(0)\nsys.exit(3)\n") % str(tmp_path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=str(tmp_path))
    assert r.returncode == 0 and "libvc.so is not built" in r.stdout, (r.returncode, r.stdout, r.stderr)
