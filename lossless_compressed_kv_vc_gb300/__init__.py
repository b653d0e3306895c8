"""Python binding of libvc, the GB300 (sm_103a) VeriCache draft/verify/accept hot path.

Argument marshalling only: every step runs in the library's CUDA kernels. The names follow the
C ABI in include/vc.h (vc_comp_bytes, vc_compress_kv, vc_draft_attn(_noalloc), vc_verify_attn(_heads), vc_accept,
vc_append_kv, vc_stage_full_kv, vc_snapkv_importance, vc_plan_stagger(_local), vc_stagger_period and the
workspace-size / status-string calls). Tensors are torch tensors on the GPU; their data pointers
and the current (or given) CUDA stream are passed through.

Importing this package loads libvc.so and raises ImportError when it has not been built
(`python -c "import __graft_entry__ as g; g.build()"`); there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libvc.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
_lib = C.CDLL(LIB_PATH)

VC_OK, VC_ERR_INVALID, VC_ERR_UNSUPPORTED, VC_ERR_CUDA, VC_ERR_NOT_PINNED, VC_ERR_WORKSPACE = range(6)
VC_DEV_OK, VC_DEV_BOUNDS, VC_DEV_TIMEOUT, VC_DEV_RANGE, VC_DEV_INTERNAL = range(5)
VC_TOKEN_DROP, VC_QUANT = 0, 1
VC_CALL_DRAFT, VC_CALL_VERIFY = 0, 1
VC_MAX_BATCH = 32
VC_APPEND_MAX_ROWS = 256
VC_STAGGER_MAX = 24
VC_STAGGER_LOCAL_MAX = 4096
VC_POOL_MAX, VC_POOL_AVG = 0, 1
VC_DRAFT_MAX_KV_HEADS = 256
VC_DRAFT_COUNTER_BYTES = VC_DRAFT_MAX_KV_HEADS * VC_MAX_BATCH * 4
VC_DRAFT_NOALLOC_SCRATCH_BYTES = 32 << 20

_p = C.c_void_p
_i32 = C.c_int32


class vc_shape(C.Structure):
    _fields_ = [("B", _i32), ("Hq", _i32), ("Hkv", _i32), ("d", _i32)]


class vc_kv_full(C.Structure):
    _fields_ = [("k", _p), ("v", _p), ("ctx", _i32), ("cap", _i32)]


class vc_kv_comp(C.Structure):
    _fields_ = [("mode", _i32), ("bits", _i32), ("keep", _i32), ("compact", _i32), ("idx", _p),
                ("k_rows", _p), ("v_rows", _p), ("rows_cap", _i32), ("ng", _i32),
                ("kc", _p), ("ks", _p), ("kz", _p), ("vc", _p), ("vs", _p), ("vz", _p),
                ("k_win", _p), ("v_win", _p), ("win_cap", _i32), ("n_win", _i32), ("ng_cap", _i32)]


class vc_draft_req(C.Structure):
    _fields_ = [("q", _p), ("k_new", _p), ("v_new", _p), ("o", _p), ("comp", vc_kv_comp)]


class vc_append_req(C.Structure):
    _fields_ = [("k_rows", _p), ("v_rows", _p), ("n_rows", _i32)]


class vc_importance_req(C.Structure):
    _fields_ = [("full", vc_kv_full), ("q_obs", _p), ("importance", _p)]


class vc_stagger_cost(C.Structure):
    _fields_ = [("draft_ns", C.c_int64), ("verify_ns", C.c_int64), ("stage_ns", C.c_int64)]


class vc_comp_sizes(C.Structure):
    _fields_ = [("ng", _i32), ("n_res", _i32), ("ng_cap", _i32), ("win_cap", _i32), ("keep", _i32), ("pad_", _i32),
                ("idx_bytes", C.c_size_t), ("rows_bytes", C.c_size_t), ("codes_bytes", C.c_size_t),
                ("kscale_bytes", C.c_size_t), ("vscale_bytes", C.c_size_t), ("win_bytes", C.c_size_t)]


class vc_verify_req(C.Structure):
    _fields_ = [("full", vc_kv_full), ("q", _p), ("k_new", _p), ("v_new", _p), ("new_cap", _i32),
                ("n_rows", _i32), ("o", _p)]


_lib.vc_compress_kv.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_kv_full), C.POINTER(_p), C.POINTER(_i32),
                                _i32, C.POINTER(vc_kv_comp), _p, _p]
_lib.vc_draft_attn.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_draft_req), _p, C.c_size_t, _p, _p]
_lib.vc_draft_attn_noalloc.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_draft_req), _p, _p]
_lib.vc_verify_attn.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_verify_req), _p, C.c_size_t, _p, _p]
_lib.vc_verify_attn_heads.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_verify_req), _i32, _i32, _p, C.c_size_t,
                                      _p, _p]
_lib.vc_verify_launches.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_verify_req)]
_lib.vc_verify_launches.restype = _i32
_lib.vc_accept.argtypes = [_i32, _i32, _i32, _p, _p, _p, _p, _p, _p]
_lib.vc_append_kv.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_kv_full), C.POINTER(vc_kv_comp),
                              C.POINTER(vc_append_req), _i32, _p, _p]
_lib.vc_stage_full_kv.argtypes = [_p, _p, C.c_size_t, C.c_size_t, _p, _p]
_lib.vc_snapkv_importance.argtypes = [C.POINTER(vc_shape), C.POINTER(vc_importance_req), _i32, _i32, _i32, _p,
                                      C.c_size_t, _p, _p]
_lib.vc_importance_workspace_size.argtypes = [C.POINTER(vc_shape), _i32, _i32]
_lib.vc_importance_workspace_size.restype = C.c_size_t
_lib.vc_plan_stagger.argtypes = [C.POINTER(vc_stagger_cost), _i32, C.POINTER(_i32), C.POINTER(C.c_int64)]
_lib.vc_stagger_period.argtypes = [C.POINTER(vc_stagger_cost), _i32, C.POINTER(_i32), C.POINTER(C.c_int64)]
_lib.vc_plan_stagger_local.argtypes = [C.POINTER(vc_stagger_cost), _i32, C.POINTER(_i32), C.POINTER(C.c_int64)]
_lib.vc_comp_bytes.argtypes = [C.POINTER(vc_shape), _i32, _i32, _i32, _i32, _i32, _i32, _i32, C.POINTER(vc_comp_sizes)]
_lib.vc_workspace_size.argtypes = [_i32, C.POINTER(vc_shape), _i32]
_lib.vc_workspace_size.restype = C.c_size_t
_lib.vc_status_string.argtypes = [_i32]
_lib.vc_status_string.restype = C.c_char_p
_lib.vc_version.restype = _i32
for _f in ("vc_compress_kv", "vc_draft_attn", "vc_draft_attn_noalloc", "vc_verify_attn", "vc_verify_attn_heads",
           "vc_accept", "vc_stage_full_kv", "vc_append_kv", "vc_plan_stagger", "vc_stagger_period",
           "vc_plan_stagger_local", "vc_snapkv_importance", "vc_comp_bytes"):
    getattr(_lib, _f).restype = _i32

EXPORTS = ["vc_compress_kv", "vc_draft_attn", "vc_draft_attn_noalloc", "vc_verify_attn", "vc_verify_attn_heads",
           "vc_accept", "vc_stage_full_kv", "vc_append_kv", "vc_plan_stagger", "vc_stagger_period",
           "vc_plan_stagger_local", "vc_snapkv_importance", "vc_importance_workspace_size", "vc_workspace_size", "vc_status_string",
           "vc_version", "vc_comp_bytes"]


class VCError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call}: {vc_status_string(status)} ({status})")
        self.status = status


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, call: str, raise_on_error: bool):
    if st != VC_OK and raise_on_error:
        raise VCError(st, call)
    return st


def vc_status_string(status: int) -> str:
    return _lib.vc_status_string(status).decode()


def vc_version() -> int:
    return _lib.vc_version()


def vc_workspace_size(call: int, shape: vc_shape, max_rows: int = 0) -> int:
    return _lib.vc_workspace_size(call, C.byref(shape), max_rows)


def vc_comp_bytes(shape: vc_shape, mode: int, bits: int, ctx: int, max_ctx: int = 0, keep: int = 0,
                  residual_min: int = 128, max_drafts: int = 0) -> vc_comp_sizes:
    """Sizes of one request's compressed-cache buffers (max_ctx 0 = ctx). Raises VCError on bad arguments."""
    out = vc_comp_sizes()
    st = _lib.vc_comp_bytes(C.byref(shape), mode, bits, ctx, max_ctx or ctx, keep, residual_min, max_drafts,
                            C.byref(out))
    _check(st, "vc_comp_bytes", True)
    return out


def vc_compress_kv(shape: vc_shape, full, importance, recent, residual_min: int, comp, dev_status=None,
                   stream=None, raise_on_error=True) -> int:
    """full: vc_kv_full array [B]; importance: list of fp32 tensors (or None for quant);
    recent: list of ints (or None); comp: vc_kv_comp array [B] (ng, n_win, keep updated in place)."""
    B = shape.B
    imp = None
    if importance is not None:
        imp = (_p * B)(*[_ptr(t) for t in importance])
    rec = None
    if recent is not None:
        rec = (_i32 * B)(*recent)
    st = _lib.vc_compress_kv(C.byref(shape), full, imp, rec, residual_min, comp, _ptr(dev_status), _stream(stream))
    return _check(st, "vc_compress_kv", raise_on_error)


def vc_draft_attn(shape: vc_shape, req, ws=None, dev_status=None, stream=None, raise_on_error=True) -> int:
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.vc_draft_attn(C.byref(shape), req, _ptr(ws), wsb, _ptr(dev_status), _stream(stream))
    return _check(st, "vc_draft_attn", raise_on_error)


def vc_draft_attn_noalloc(shape: vc_shape, req, dev_status=None, stream=None, raise_on_error=True) -> int:
    """vc_draft_attn with the library's built-in scratch instead of a caller workspace (allocates nothing)."""
    st = _lib.vc_draft_attn_noalloc(C.byref(shape), req, _ptr(dev_status), _stream(stream))
    return _check(st, "vc_draft_attn_noalloc", raise_on_error)


def vc_verify_attn(shape: vc_shape, req, ws=None, dev_status=None, stream=None, raise_on_error=True) -> int:
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.vc_verify_attn(C.byref(shape), req, _ptr(ws), wsb, _ptr(dev_status), _stream(stream))
    return _check(st, "vc_verify_attn", raise_on_error)


def vc_verify_attn_heads(shape: vc_shape, req, kv_head_begin: int, kv_head_end: int, ws=None, dev_status=None,
                         stream=None, raise_on_error=True) -> int:
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.vc_verify_attn_heads(C.byref(shape), req, kv_head_begin, kv_head_end, _ptr(ws), wsb, _ptr(dev_status),
                                   _stream(stream))
    return _check(st, "vc_verify_attn_heads", raise_on_error)


def vc_verify_launches(shape: vc_shape, req) -> int:
    """Kernels one vc_verify_attn call launches for these requests (host only; -1: invalid)."""
    return int(_lib.vc_verify_launches(C.byref(shape), req))


def vc_accept(B: int, L_max: int, V: int, logits, draft, L, out_tokens, n_acc, stream=None,
              raise_on_error=True) -> int:
    st = _lib.vc_accept(B, L_max, V, _ptr(logits), _ptr(draft), _ptr(L), _ptr(out_tokens), _ptr(n_acc),
                        _stream(stream))
    return _check(st, "vc_accept", raise_on_error)


def vc_append_kv(shape: vc_shape, full, comp, req, residual_min: int, dev_status=None, stream=None,
                 raise_on_error=True) -> int:
    """full: vc_kv_full array [B] (ctx updated in place); comp: vc_kv_comp array [B] (ng, n_win
    updated in place for VC_QUANT); req: vc_append_req array [B]."""
    st = _lib.vc_append_kv(C.byref(shape), full, comp, req, residual_min, _ptr(dev_status), _stream(stream))
    return _check(st, "vc_append_kv", raise_on_error)


def vc_stage_full_kv(host_src, dev_dst, nbytes: int, chunk_bytes: int = 0, copy_stream=None, done=None,
                     raise_on_error=True) -> int:
    ev = done.cuda_event if done is not None and not isinstance(done, int) else done
    st = _lib.vc_stage_full_kv(_ptr(host_src), _ptr(dev_dst), nbytes, chunk_bytes, _stream(copy_stream), ev)
    return _check(st, "vc_stage_full_kv", raise_on_error)


def vc_importance_workspace_size(shape: vc_shape, window: int, max_ctx: int) -> int:
    return _lib.vc_importance_workspace_size(C.byref(shape), window, max_ctx)


def vc_snapkv_importance(shape: vc_shape, req, window: int, pool_kernel: int = 7, pool_kind: int = VC_POOL_MAX,
                         ws=None, dev_status=None, stream=None, raise_on_error=True) -> int:
    """req: vc_importance_req array [B]; writes each request's importance [ctx]."""
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    st = _lib.vc_snapkv_importance(C.byref(shape), req, window, pool_kernel, pool_kind, _ptr(ws), wsb,
                                   _ptr(dev_status), _stream(stream))
    return _check(st, "vc_snapkv_importance", raise_on_error)


def _costs(costs):
    """costs: sequence of (draft_ns, verify_ns, stage_ns) integers."""
    arr = (vc_stagger_cost * len(costs))()
    for r, (d, v, s) in enumerate(costs):
        arr[r].draft_ns, arr[r].verify_ns, arr[r].stage_ns = int(d), int(v), int(s)
    return arr


def vc_plan_stagger(costs, raise_on_error=True):
    """Exact two-group split of cross-resource staggering. Returns (status, groups list, period_ns)."""
    n = len(costs)
    grp = (_i32 * max(n, 1))()
    t = C.c_int64(0)
    st = _lib.vc_plan_stagger(_costs(costs) if n else None, n, grp, C.byref(t))
    _check(st, "vc_plan_stagger", raise_on_error)
    return st, list(grp)[:n], t.value


def vc_plan_stagger_local(costs, raise_on_error=True):
    """Local-search two-group split for any batch up to VC_STAGGER_LOCAL_MAX requests (no
    optimality guarantee). Returns (status, groups list, period_ns)."""
    n = len(costs)
    grp = (_i32 * max(n, 1))()
    t = C.c_int64(0)
    st = _lib.vc_plan_stagger_local(_costs(costs) if n else None, n, grp, C.byref(t))
    _check(st, "vc_plan_stagger_local", raise_on_error)
    return st, list(grp)[:n], t.value


def vc_stagger_period(costs, groups, raise_on_error=True):
    n = len(costs)
    grp = (_i32 * max(n, 1))(*groups)
    t = C.c_int64(0)
    st = _lib.vc_stagger_period(_costs(costs) if n else None, n, grp, C.byref(t))
    _check(st, "vc_stagger_period", raise_on_error)
    return st, t.value


def lib_handle():
    return _lib
