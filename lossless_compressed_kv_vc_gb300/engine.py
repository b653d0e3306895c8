"""Per-request buffers and descriptors for one batch of VeriCache requests on one GPU.

A `Batch` owns the device tensors a round needs (full cache, compressed cache, window, outputs)
and fills the vc.h descriptors that point at them; its methods are one C-ABI call each:
compress -> L x draft_step -> verify -> accept, then append_accepted to carry the accepted tokens
into the next round ("VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core
algorithm"). torch is used for memory and streams only.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

from . import (vc_shape, vc_kv_full, vc_kv_comp, vc_draft_req, vc_verify_req, vc_append_req, vc_importance_req,
               vc_snapkv_importance, vc_importance_workspace_size, VC_POOL_MAX, vc_compress_kv, vc_comp_bytes,
               vc_draft_attn, vc_verify_attn, vc_verify_attn_heads, vc_verify_launches, vc_accept, vc_append_kv, vc_workspace_size,
               VC_TOKEN_DROP, VC_QUANT, VC_CALL_DRAFT, VC_CALL_VERIFY)


@dataclass
class Req:
    mode: int
    ctx: int
    L: int
    k_full: torch.Tensor            # bf16 [Hkv][cap][d] (device, or the staging buffer)
    v_full: torch.Tensor
    q: torch.Tensor                 # bf16 [L][Hq][d]
    k_new: torch.Tensor             # bf16 [L][Hkv][d]
    v_new: torch.Tensor
    importance: Optional[torch.Tensor] = None
    keep: int = 0
    recent: int = 0
    compact: bool = False
    bits: int = 2
    grow: int = 0                   # tokens the context may gain through append_accepted
    # owned buffers
    idx: Optional[torch.Tensor] = None
    k_rows: Optional[torch.Tensor] = None
    v_rows: Optional[torch.Tensor] = None
    kc: Optional[torch.Tensor] = None
    ks: Optional[torch.Tensor] = None
    kz: Optional[torch.Tensor] = None
    vc: Optional[torch.Tensor] = None
    vs: Optional[torch.Tensor] = None
    vz: Optional[torch.Tensor] = None
    k_win: Optional[torch.Tensor] = None
    v_win: Optional[torch.Tensor] = None
    o_draft: Optional[torch.Tensor] = None   # bf16 [L][Hq][d]
    o_verify: Optional[torch.Tensor] = None  # bf16 [L][Hq][d]
    n_res: int = 0


class Batch:
    """Requests of one compression mode that draft together (<= 32 per C-ABI call)."""

    def __init__(self, Hq: int, Hkv: int, d: int, reqs: List[Req], residual_min: int = 128, device="cuda"):
        assert len(reqs) >= 1
        self.Hq, self.Hkv, self.d = Hq, Hkv, d
        self.reqs = reqs
        self.residual_min = residual_min
        self.device = device
        self.shape = vc_shape(len(reqs), Hq, Hkv, d)
        self.L_max = max(r.L for r in reqs)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)
        for r in reqs:
            self._alloc(r)
        self.full = (vc_kv_full * len(reqs))()
        self.comp = (vc_kv_comp * len(reqs))()
        for b, r in enumerate(reqs):
            self._fill(b, r)
        # zero-filled once: the draft call's arrival counters start at zero and return to zero
        self.ws_draft = torch.zeros(vc_workspace_size(VC_CALL_DRAFT, self.shape) // 4 + 64, dtype=torch.float32,
                                    device=device)
        vb = vc_workspace_size(VC_CALL_VERIFY, self.shape, self.L_max)
        self.ws_verify = torch.empty(max(vb // 4 + 64, 64), dtype=torch.float32, device=device)
        # The zero fills above run on the current stream; a call this Batch issues on another
        # stream (a compress writing the windows, a draft reading the counters) must follow them,
        # so each stream it is given waits for this event once, before its first call.
        self._built = torch.cuda.Event()
        self._built.record()
        self._ordered = set()

    def _order(self, *streams):
        for s in streams:
            if s is None:
                continue
            if not isinstance(s, torch.cuda.Stream):
                s = torch.cuda.ExternalStream(int(s))
            if s.cuda_stream not in self._ordered:
                s.wait_event(self._built)
                self._ordered.add(s.cuda_stream)

    def _alloc(self, r: Req):
        """Buffers of one request, sized by the library's own layout query (vc_comp_bytes): the
        residual and block counts, the block capacity for a context grown by r.grow tokens and the
        window rows are the library's rules, not restated here."""
        Hkv, d, dev = self.Hkv, self.d, self.device
        sz = vc_comp_bytes(vc_shape(1, self.Hq, Hkv, d), r.mode, r.bits, r.ctx, r.ctx + r.grow, r.keep,
                           self.residual_min, r.L)
        if r.mode == VC_TOKEN_DROP:
            keep = sz.keep
            r.idx = torch.empty(sz.idx_bytes // 4, dtype=torch.int32, device=dev)
            if r.compact:
                r.k_rows = torch.empty((Hkv, keep, d), dtype=torch.bfloat16, device=dev)
                r.v_rows = torch.empty((Hkv, keep, d), dtype=torch.bfloat16, device=dev)
            r.n_res = 0
        else:
            r.n_res = sz.n_res
            ng_cap = sz.ng_cap
            u8, f16 = torch.uint8, torch.float16
            r.kc = torch.empty((Hkv, ng_cap, sz.codes_bytes // (Hkv * ng_cap)), dtype=u8, device=dev)
            r.ks = torch.empty((Hkv, ng_cap, d), dtype=f16, device=dev)
            r.kz = torch.empty((Hkv, ng_cap, d), dtype=f16, device=dev)
            r.vc = torch.empty((Hkv, ng_cap, sz.codes_bytes // (Hkv * ng_cap)), dtype=u8, device=dev)
            r.vs = torch.empty((Hkv, sz.vscale_bytes // (2 * Hkv * (d // 32)), d // 32), dtype=f16, device=dev)
            r.vz = torch.empty((Hkv, sz.vscale_bytes // (2 * Hkv * (d // 32)), d // 32), dtype=f16, device=dev)
        win_cap = sz.win_cap
        r.k_win = torch.zeros((Hkv, win_cap, d), dtype=torch.bfloat16, device=dev)
        r.v_win = torch.zeros((Hkv, win_cap, d), dtype=torch.bfloat16, device=dev)
        r.o_draft = torch.empty((r.L, self.Hq, d), dtype=torch.bfloat16, device=dev)
        r.o_verify = torch.empty((r.L, self.Hq, d), dtype=torch.bfloat16, device=dev)

    def _fill(self, b: int, r: Req):
        f = self.full[b]
        f.k, f.v = r.k_full.data_ptr(), r.v_full.data_ptr()
        f.ctx, f.cap = r.ctx, r.k_full.shape[1]
        c = self.comp[b]
        c.mode = r.mode
        c.bits = r.bits
        if r.mode == VC_TOKEN_DROP:
            c.keep = r.keep
            c.compact = int(r.compact)
            c.idx = r.idx.data_ptr()
            if r.compact:
                c.k_rows, c.v_rows, c.rows_cap = r.k_rows.data_ptr(), r.v_rows.data_ptr(), r.k_rows.shape[1]
        else:
            c.kc, c.ks, c.kz = r.kc.data_ptr(), r.ks.data_ptr(), r.kz.data_ptr()
            c.vc, c.vs, c.vz = r.vc.data_ptr(), r.vs.data_ptr(), r.vz.data_ptr()
            c.ng_cap = r.kc.shape[1]
        c.k_win, c.v_win, c.win_cap = r.k_win.data_ptr(), r.v_win.data_ptr(), r.k_win.shape[1]

    def set_full(self, b: int, k: torch.Tensor, v: torch.Tensor):
        """Point request b's KV_full at other device tensors (e.g. a staging buffer)."""
        r = self.reqs[b]
        r.k_full, r.v_full = k, v
        f = self.full[b]
        f.k, f.v, f.cap = k.data_ptr(), v.data_ptr(), k.shape[1]

    # ---- the round's calls -------------------------------------------------------------------
    def snapkv_importance(self, q_obs, window: int, pool_kernel: int = 7, pool_kind: int = VC_POOL_MAX, stream=None):
        """Fill every token-drop request's importance from its observation window (SnapKV style,
        vc_snapkv_importance): q_obs[b] is request b's bf16 [window][Hq][d] queries of its last
        `window` context tokens. The next compress selects the keep-set from it."""
        drop = [b for b, r in enumerate(self.reqs) if r.mode == VC_TOKEN_DROP]
        if not drop:
            return
        arr = (vc_importance_req * len(drop))()
        for i, b in enumerate(drop):
            arr[i].full = self.full[b]
            arr[i].q_obs = q_obs[b].data_ptr()
            arr[i].importance = self.reqs[b].importance.data_ptr()
        shape = vc_shape(len(drop), self.Hq, self.Hkv, self.d)
        need = vc_importance_workspace_size(shape, window, max(self.reqs[b].ctx for b in drop))
        ws = getattr(self, "ws_importance", None)
        if ws is None or ws.numel() * 4 < need:
            ws = self.ws_importance = torch.empty(need // 4 + 64, dtype=torch.float32, device=self.device)
        self._order(stream)
        vc_snapkv_importance(shape, arr, window, pool_kernel, pool_kind, ws, self.dev_status, stream)

    def compress(self, stream=None, importance=None):
        self._order(stream)
        mode = self.reqs[0].mode
        if mode == VC_TOKEN_DROP:
            imp = importance if importance is not None else [r.importance for r in self.reqs]
            vc_compress_kv(self.shape, self.full, imp, [r.recent for r in self.reqs],
                           self.residual_min, self.comp, self.dev_status, stream)
        else:
            vc_compress_kv(self.shape, self.full, None, None, self.residual_min, self.comp, self.dev_status, stream)

    def reset_window(self):
        for b, r in enumerate(self.reqs):
            self.comp[b].n_win = r.n_res

    def draft_requests(self, step: int):
        """vc_draft_req array for step `step` over the requests whose L exceeds it."""
        act = [b for b, r in enumerate(self.reqs) if step < r.L]
        arr = (vc_draft_req * len(act))()
        for i, b in enumerate(act):
            r = self.reqs[b]
            e = arr[i]
            e.q = r.q[step].data_ptr()
            e.k_new = r.k_new[step].data_ptr()
            e.v_new = r.v_new[step].data_ptr()
            e.o = r.o_draft[step].data_ptr()
            e.comp = self.comp[b]
        return act, arr

    def draft_step(self, step: int, stream=None):
        act, arr = self.draft_requests(step)
        if not act:
            return
        shape = vc_shape(len(act), self.Hq, self.Hkv, self.d)
        self._order(stream)
        vc_draft_attn(shape, arr, self.ws_draft, self.dev_status, stream)
        for b in act:
            self.comp[b].n_win += 1

    def prepare_steps(self):
        """Descriptor arrays of every draft step of a round (window counts as after compress), so
        a round issues its calls without rebuilding them. Call it after the first compress: the
        arrays copy the compressed-cache descriptors, whose sizes compress fills in."""
        self._steps = []
        self._verify_arr = self.verify_requests()
        for s in range(self.L_max):
            act, arr = self.draft_requests(s)
            for i, b in enumerate(act):
                arr[i].comp.n_win = self.reqs[b].n_res + s
            self._steps.append((vc_shape(len(act), self.Hq, self.Hkv, self.d), arr, act))

    def run_round(self, logits, draft, L, out_tokens, n_acc, stream=None, draft_events=None, compress=True):
        """compress -> L_max draft steps -> verify -> accept, all on `stream`. draft_events, if
        given, is a (start, end) pair of CUDA events recorded around the whole draft phase (an
        event between two draft steps would hold back the next step's early start). compress=False
        drafts from the caches as they stand (quantised caches kept current by append_accepted)."""
        self._order(stream)
        if compress:
            self.compress(stream)
        if draft_events is not None:
            draft_events[0].record(stream)
        for s, (shape, arr, act) in enumerate(self._steps):
            vc_draft_attn(shape, arr, self.ws_draft, self.dev_status, stream)
        if draft_events is not None:
            draft_events[1].record(stream)
        vc_verify_attn(self.shape, self._verify_arr, self.ws_verify, self.dev_status, stream)
        accept(logits, draft, L, out_tokens, n_acc, stream)

    def run_round_from_host(self, hr: "HostRound", stream, copy_stream, draft_events=None, compress=True):
        """One round whose inputs sit in pinned host memory and whose results go back to it.

        All of the round's inputs cross the host link on `copy_stream` into the next of the
        HostRound's device slots, once that slot's previous round has accepted: the draft inputs
        (queries, drafted K/V, importance) first, then the accept inputs (drafts, logits, L). The
        compute stream waits for the draft inputs before compress and for the accept inputs before
        accept, so the largest transfer of a round (the logits) hides under the HBM-bound draft
        phase ("Cross-resource staggering (P1)": keep the host link busy while the GPU drafts),
        and with two slots a round's copies overlap the previous round on the GPU."""
        self._order(stream, copy_stream)
        sl = hr.next_slot()
        copy_stream.wait_event(sl.free)
        with torch.cuda.stream(copy_stream):
            for h, d in zip(hr.draft_host, sl.draft_dev):
                d.copy_(h, non_blocking=True)
        sl.ready.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            for h, d in zip(hr.accept_host, sl.accept_dev):
                d.copy_(h, non_blocking=True)
        sl.landed.record(copy_stream)
        stream.wait_event(sl.ready)
        if compress:
            self.compress(stream, importance=sl.importance)
        if draft_events is not None:
            draft_events[0].record(stream)
        for shape, arr, act in sl.steps:
            vc_draft_attn(shape, arr, self.ws_draft, self.dev_status, stream)
        if draft_events is not None:
            draft_events[1].record(stream)
        vc_verify_attn(self.shape, sl.verify_arr, self.ws_verify, self.dev_status, stream)
        stream.wait_event(sl.landed)
        draft, logits, L = sl.accept_dev
        accept(logits, draft, L, hr.out_tokens, hr.n_acc, stream)
        sl.free.record(stream)
        with torch.cuda.stream(stream):
            hr.host_tokens.copy_(hr.out_tokens, non_blocking=True)
            hr.host_n_acc.copy_(hr.n_acc, non_blocking=True)

    def append_accepted(self, n_acc, stream=None):
        """Carry a round's accepted drafts into the caches ("Core algorithm": the next round
        starts after the last accepted token). n_acc: host sequence of accepted counts per request
        (accepted drafts + the bonus/correction token). The n_acc - 1 accepted drafts' K/V (this
        round's k_new/v_new rows) are appended to KV_full and, for quantised requests, the blocks
        that became whole are quantised and the window restarts with the new residual. The bonus
        token's K/V belongs to the next round. The round's descriptor arrays are rebuilt."""
        arr = (vc_append_req * len(self.reqs))()
        for b, r in enumerate(self.reqs):
            n = max(0, min(int(n_acc[b]) - 1, r.L))
            arr[b].k_rows, arr[b].v_rows, arr[b].n_rows = r.k_new.data_ptr(), r.v_new.data_ptr(), n
        self._order(stream)
        vc_append_kv(self.shape, self.full, self.comp, arr, self.residual_min, self.dev_status, stream)
        for b, r in enumerate(self.reqs):
            r.ctx = self.full[b].ctx
            if r.mode == VC_QUANT:
                r.n_res = self.comp[b].n_win  # the window restarts with the new residual
        if getattr(self, "_steps", None) is not None:
            self.prepare_steps()

    def verify_requests(self):
        arr = (vc_verify_req * len(self.reqs))()
        for b, r in enumerate(self.reqs):
            e = arr[b]
            e.full = self.full[b]
            e.q = r.q.data_ptr()
            e.k_new = r.k_win.data_ptr() + r.n_res * self.d * 2
            e.v_new = r.v_win.data_ptr() + r.n_res * self.d * 2
            e.new_cap = r.k_win.shape[1]
            e.n_rows = r.L
            e.o = r.o_verify.data_ptr()
        return arr

    def verify(self, stream=None):
        self._order(stream)
        vc_verify_attn(self.shape, self.verify_requests(), self.ws_verify, self.dev_status, stream)

    def verify_launches(self) -> int:
        """Kernels one verify() launches for this batch (the library's own split of its KV heads by
        row tiles, under the current environment switches)."""
        return vc_verify_launches(self.shape, self.verify_requests())


class _Slot:
    """One set of device input buffers of a HostRound with the descriptor arrays that point at
    them, and its events: ready (draft inputs landed), landed (accept inputs landed), free (the
    slot's last round has accepted)."""

    def __init__(self, draft_dev, accept_dev, importance, steps, verify_arr, stream):
        self.draft_dev, self.accept_dev, self.importance = draft_dev, accept_dev, importance
        self.steps, self.verify_arr = steps, verify_arr
        self.ready, self.landed, self.free = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        self.free.record(stream)


class HostRound:
    """Pinned host buffers of one round's inputs and results, and `slots` sets of device buffers
    they land in, used round-robin (the first is the batch's own tensors).

    Inputs: each request's queries, drafted K/V rows and (token drop) importance, which the draft
    phase reads, and the batch's drafts [B][L_max], logits [B][L_max+1][V] and L [B], which only
    accept reads. Results: accepted tokens [B][L_max+1] and counts [B], valid on the host once the
    round's stream has been synchronised. Build it after the batch's first compress (it rebuilds
    the batch's descriptor arrays for every slot)."""

    def __init__(self, bt: Batch, logits: torch.Tensor, draft: torch.Tensor, L: torch.Tensor,
                 out_tokens: torch.Tensor, n_acc: torch.Tensor, slots: int = 2,
                 names=("q", "k_new", "v_new", "importance")):
        """names: the per-request inputs the round reads and so copies (importance only when the
        round compresses)."""
        pin = lambda t: t.detach().to("cpu").pin_memory()
        fields = [(r, n) for r in bt.reqs for n in names if getattr(r, n) is not None]
        self.draft_host = [pin(getattr(r, n)) for r, n in fields]
        self.accept_host = [pin(t) for t in (draft, logits, L)]
        self.accept_inputs = list(zip(self.accept_host, (draft, logits, L)))
        self.out_tokens, self.n_acc = out_tokens, n_acc
        self.host_tokens = torch.empty(out_tokens.shape, dtype=out_tokens.dtype).pin_memory()
        self.host_n_acc = torch.empty(n_acc.shape, dtype=n_acc.dtype).pin_memory()
        stream = torch.cuda.current_stream()
        self.slots = []
        own = [getattr(r, n) for r, n in fields]
        for s in range(slots):
            dev = own if s == 0 else [torch.empty_like(t) for t in own]
            acc = [draft, logits, L] if s == 0 else [torch.empty_like(t) for t in (draft, logits, L)]
            for (r, n), t in zip(fields, dev):  # build this slot's descriptor arrays
                setattr(r, n, t)
            bt.prepare_steps()
            imp = [r.importance for r in bt.reqs]
            self.slots.append(_Slot(dev, acc, imp, bt._steps, bt._verify_arr, stream))
        for (r, n), t in zip(fields, own):
            setattr(r, n, t)
        bt.prepare_steps()
        self._next = 0

    def next_slot(self) -> _Slot:
        sl = self.slots[self._next]
        self._next = (self._next + 1) % len(self.slots)
        return sl

    @property
    def h2d_bytes(self) -> int:
        return sum(h.numel() * h.element_size() for h in self.draft_host + self.accept_host)

    @property
    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.host_tokens, self.host_n_acc))


def accept(logits: torch.Tensor, draft: torch.Tensor, L: torch.Tensor, out_tokens=None, n_acc=None, stream=None):
    B, Lp1, V = logits.shape
    if out_tokens is None:
        out_tokens = torch.empty((B, Lp1), dtype=torch.int32, device=logits.device)
    if n_acc is None:
        n_acc = torch.empty((B,), dtype=torch.int32, device=logits.device)
    vc_accept(B, Lp1 - 1, V, logits, draft, L, out_tokens, n_acc, stream)
    return out_tokens, n_acc


class StaggeredOffload:
    """Cross-resource staggering for requests whose KV_full lives in pinned host memory
    ("VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Cross-resource staggering
    (P1)" and "Architecture support", long-context decoding).

    Two groups of requests alternate roles. In each phase one group drafts its L steps on the
    compute stream (HBM-bound) while the other group's KV_full is copied host-to-device on the copy
    stream (host-link-bound); the compute stream then waits for that copy and verifies and accepts
    the staged group. Each request keeps its own device staging slot, so a copy never waits for the
    other group's verification.

    A group is one Batch or a list of Batches (one per compression mode: a batch that mixes token
    drop and quantisation drafts with one C-ABI call per mode); host_kv[g] and slots[g] list the
    group's requests in that order (batch by batch). host_kv[g][i] (pinned [K; V] buffer) and
    slots[g][i] (its device copy, which the request's KV_full descriptor points at) are None for a
    request whose KV_full stays in HBM; such a request drafts and verifies in its group's phases
    with nothing to copy. plan_groups chooses the groups.

    head_chunks > 1 pipelines the copy into the verification ("Cross-resource staggering (P1)"
    applied to the verification itself): a group's KV_full is copied a range of KV heads at a time
    (each head's K and V rows are contiguous in the [K; V][Hkv][cap][d] layout), each range records
    its own event, and the compute stream verifies each head range (vc_verify_attn_heads) as soon as
    it has landed, so only the last range's verification remains once the copy ends.
    """

    def __init__(self, groups, host_kv: List[List[Optional[torch.Tensor]]],
                 slots: List[List[Optional[torch.Tensor]]],
                 copy_stream, compute_stream, chunk_bytes: int = 64 << 20, head_chunks: int = 1):
        assert len(groups) == 2
        self.groups = [list(g) if isinstance(g, (list, tuple)) else [g] for g in groups]
        self.single = [not isinstance(g, (list, tuple)) for g in groups]
        Hkv = self.groups[0][0].Hkv
        assert 1 <= head_chunks <= Hkv and all(bt.Hkv == Hkv for grp in self.groups for bt in grp)
        for g in range(2):
            assert len(host_kv[g]) == len(slots[g]) == sum(len(bt.reqs) for bt in self.groups[g])
        self.host_kv, self.slots = host_kv, slots
        self.copy_stream, self.compute_stream = copy_stream, compute_stream
        self.chunk_bytes = chunk_bytes
        self.edges = [c * Hkv // head_chunks for c in range(head_chunks + 1)]
        self.staged = [[torch.cuda.Event() for _ in range(head_chunks)] for _ in range(2)]
        self.verified = [torch.cuda.Event(), torch.cuda.Event()]
        # the batches, slots and round tensors were made on the current stream: both streams
        # start after that work
        cur = torch.cuda.current_stream()
        copy_stream.wait_stream(cur)
        compute_stream.wait_stream(cur)
        for g in range(2):  # a slot is free before its first copy
            self.verified[g].record(compute_stream)
        self._cur = [None, None]  # host-input periods: the HostRound slot each batch last drafted from
        self._graphs = {}  # (id of a descriptor-array list) -> CUDA graph of that draft series

    def capture_drafts(self, host_rounds=None):
        """Capture each batch's draft series (its L_max vc_draft_attn calls, one per step, with the
        descriptor arrays they use in a period: the batch's own, and those of each HostRound slot
        when host_rounds is given) as a CUDA graph on the compute stream; phase() then replays the
        graph instead of issuing the calls one by one. The calls are the same kernels with the same
        arguments (the arrays are fixed per step); a replay costs the host one launch instead of
        L_max C-ABI calls, so the host keeps ahead of the GPU. Call it after a first period (the
        kernels' one-time set-up has run) and before the timed ones."""
        ks = self.compute_stream
        series = []
        for grp in self.groups:
            for bt in grp:
                series.append((bt, bt._steps))
        if host_rounds is not None:
            for g in range(2):
                for j, hr in enumerate(host_rounds[g]):
                    for sl in hr.slots:
                        series.append((self.groups[g][j], sl.steps))
        torch.cuda.synchronize()
        for bt, steps in series:
            if id(steps) in self._graphs:
                continue
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=ks):
                for shape, arr, act in steps:
                    vc_draft_attn(shape, arr, bt.ws_draft, bt.dev_status, ks)
            self._graphs[id(steps)] = (graph, steps)
        torch.cuda.synchronize()

    def _draft(self, bt, steps):
        """The batch's draft series on the compute stream: a graph replay when captured."""
        ks = self.compute_stream
        got = self._graphs.get(id(steps))
        if got is not None and got[1] is steps:
            with torch.cuda.stream(ks):
                got[0].replay()
            return
        for shape, arr, act in steps:
            vc_draft_attn(shape, arr, bt.ws_draft, bt.dev_status, ks)

    def stage_bytes(self, g: int) -> int:
        return sum(h.numel() * h.element_size() for h in self.host_kv[g] if h is not None)

    def stage(self, g: int, events=None):
        """Issue the host-to-device copies of group g's KV_full on the copy stream, one KV-head range
        at a time (K then V rows of those heads, for every host-resident request of the group)."""
        from . import vc_stage_full_kv
        self.copy_stream.wait_event(self.verified[g])  # its previous verification has read the slot
        if events is not None:
            events[0].record(self.copy_stream)
        for c in range(len(self.edges) - 1):
            h0, h1 = self.edges[c], self.edges[c + 1]
            for h, d in zip(self.host_kv[g], self.slots[g]):
                if h is None:  # this request's KV_full stays in HBM
                    continue
                for kv in range(2):
                    src, dst = h[kv, h0:h1], d[kv, h0:h1]
                    vc_stage_full_kv(src, dst, src.numel() * src.element_size(), self.chunk_bytes, self.copy_stream,
                                     None)
            self.staged[g][c].record(self.copy_stream)
        if events is not None:
            events[1].record(self.copy_stream)

    def _io(self, io, g):
        return [io[g]] if self.single[g] else list(io[g])

    def phase(self, draft_g: int, io, draft_events=None, stage_events=None, verify_event=None, host_rounds=None,
              verify_events=None):
        """Group draft_g drafts while the other group stages, then the other group verifies and
        accepts. io[g] = (logits, draft, L, out_tokens, n_acc) of group g's single batch, or a list
        of such tuples, one per batch of the group. draft_events: a (start, end) pair around the
        draft phase, or a list of pairs, one per batch; verify_events: a (start, end) pair around the
        other group's verification; verify_event (legacy) is recorded once it is verified.

        host_rounds[g][j] (a HostRound of batch j of group g; io is then ignored): the drafting
        group's round inputs are first copied from pinned host memory on the copy stream (its query
        and drafted K/V rows before the other group's KV_full, its drafts, logits and L after it: they
        are read only when it is verified, in the next phase), and the verified group's accepted
        tokens and counts go back to pinned host memory."""
        other = 1 - draft_g
        cs, ks = self.copy_stream, self.compute_stream
        dgrp, ogrp = self.groups[draft_g], self.groups[other]
        if host_rounds is not None:
            sls = []
            for hr in host_rounds[draft_g]:
                sl = hr.next_slot()
                cs.wait_event(sl.free)
                with torch.cuda.stream(cs):
                    for h, d in zip(hr.draft_host, sl.draft_dev):
                        d.copy_(h, non_blocking=True)
                sl.ready.record(cs)
                sls.append(sl)
            self._cur[draft_g] = sls
        self.stage(other, stage_events)
        if host_rounds is not None:
            for hr, sl in zip(host_rounds[draft_g], self._cur[draft_g]):
                with torch.cuda.stream(cs):
                    for h, d in zip(hr.accept_host, sl.accept_dev):
                        d.copy_(h, non_blocking=True)
                sl.landed.record(cs)
        per_batch = isinstance(draft_events, (list, tuple)) and len(draft_events) == len(dgrp) and \
            isinstance(draft_events[0], (list, tuple))
        if draft_events is not None and not per_batch:
            draft_events[0].record(ks)
        for j, bt in enumerate(dgrp):
            steps = bt._steps
            if host_rounds is not None:
                sl = self._cur[draft_g][j]
                ks.wait_event(sl.ready)
                steps = sl.steps
            if per_batch:
                draft_events[j][0].record(ks)
            self._draft(bt, steps)
            if per_batch:
                draft_events[j][1].record(ks)
        if draft_events is not None and not per_batch:
            draft_events[1].record(ks)
        if verify_events is not None:
            verify_events[0].record(ks)
        for c in range(len(self.edges) - 1):
            ks.wait_event(self.staged[other][c])
            for j, ob in enumerate(ogrp):
                varr = ob._verify_arr
                if host_rounds is not None and self._cur[other] is not None:
                    varr = self._cur[other][j].verify_arr
                vc_verify_attn_heads(ob.shape, varr, self.edges[c], self.edges[c + 1], ob.ws_verify,
                                     ob.dev_status, ks)
        self.verified[other].record(ks)
        if verify_events is not None:
            verify_events[1].record(ks)
        if verify_event is not None:
            verify_event.record(ks)
        if host_rounds is not None:
            for j, hr in enumerate(host_rounds[other]):
                sl = self._cur[other][j] if self._cur[other] is not None else hr.slots[0]
                ks.wait_event(sl.landed)
                dr, lg, Lt = sl.accept_dev
                accept(lg, dr, Lt, hr.out_tokens, hr.n_acc, ks)
                sl.free.record(ks)
                with torch.cuda.stream(ks):
                    hr.host_tokens.copy_(hr.out_tokens, non_blocking=True)
                    hr.host_n_acc.copy_(hr.n_acc, non_blocking=True)
            return
        for lg, dr, L, tok, nacc in self._io(io, other):
            accept(lg, dr, L, tok, nacc, ks)

    def period(self, io, events=None, host_rounds=None):
        """Both phases: every request drafts once and is verified once. events: optional dict with
        draft0/draft1 (a pair, or a list of pairs, one per batch of the group), stage0/stage1,
        verify0/verify1 (pairs) and verified0/verified1 (single events)."""
        ev = events or {}
        self.phase(0, io, ev.get("draft0"), ev.get("stage1"), ev.get("verified1"), host_rounds, ev.get("verify1"))
        self.phase(1, io, ev.get("draft1"), ev.get("stage0"), ev.get("verified0"), host_rounds, ev.get("verify0"))


def stagger_costs(draft_ns, verify_ns, stage_ns):
    """(draft, verify, stage) integer nanoseconds per request, as vc_plan_stagger takes them."""
    return [(int(round(d)), int(round(v)), int(round(s))) for d, v, s in zip(draft_ns, verify_ns, stage_ns)]


def plan_groups(costs):
    """Split requests into the two alternating groups of StaggeredOffload by the library's planner:
    exact (vc_plan_stagger) up to VC_STAGGER_MAX requests, local search (vc_plan_stagger_local)
    beyond. Returns ([indices of group 0], [indices of group 1], period_ns)."""
    from . import vc_plan_stagger, vc_plan_stagger_local, VC_STAGGER_MAX
    plan = vc_plan_stagger if len(costs) <= VC_STAGGER_MAX else vc_plan_stagger_local
    st, groups, t = plan(costs)
    return [r for r, g in enumerate(groups) if g == 0], [r for r, g in enumerate(groups) if g == 1], t


def staggered_groups(Hq: int, Hkv: int, d: int, reqs: List[Req], split, on_host, residual_min: int = 128,
                     device="cuda", stream=None):
    """The two groups of StaggeredOffload for a batch that mixes compression modes and residencies:
    request r goes to group split[r]; each group holds one Batch per compression mode (a draft call
    serves one mode); every Batch compresses (KV_comp is built once per request, while KV_full is
    still in HBM); then the KV_full of the requests with on_host[r] moves to pinned host memory,
    each with a device staging slot. A token-drop request whose KV_full leaves HBM must keep its
    kept rows in a compact copy (Req.compact). Returns (groups, members, host_kv, slots): groups[g]
    the Batches of group g, members[g][j] the request indices of its Batch j, host_kv[g] / slots[g]
    flat over the group's requests in batch order (None for HBM-resident requests)."""
    groups, members, host_kv, slots = [], [], [], []
    modes = sorted({r.mode for r in reqs})
    for gi in (0, 1):
        bts, mem = [], []
        for m in modes:
            idx = [i for i, r in enumerate(reqs) if split[i] == gi and r.mode == m]
            if not idx:
                continue
            for i in idx:
                assert m != VC_TOKEN_DROP or reqs[i].compact or not on_host[i], \
                    "a token-drop request with KV_full on the host needs compact kept rows"
            bt = Batch(Hq, Hkv, d, [reqs[i] for i in idx], residual_min=residual_min, device=device)
            bt.compress(stream)
            bts.append(bt)
            mem.append(idx)
        groups.append(bts)
        members.append(mem)
    torch.cuda.synchronize()
    for gi in (0, 1):
        h, sl = move_some_full_kv_to_host(groups[gi], [[on_host[i] for i in idx] for idx in members[gi]])
        host_kv.append(h)
        slots.append(sl)
        for bt in groups[gi]:
            bt.prepare_steps()
    return groups, members, host_kv, slots


def group_io(members, logits: torch.Tensor, draft: torch.Tensor, L: torch.Tensor):
    """Per group, per Batch: (logits, draft, L, out_tokens, n_acc) of the Batch's requests, the
    first three gathered from the whole batch's tensors."""
    io = []
    for mem in members:
        row = []
        for idx in mem:
            sel = torch.tensor(idx, device=logits.device)
            row.append((logits[sel].contiguous(), draft[sel].contiguous(), L[sel].contiguous(),
                        torch.empty((len(idx), logits.shape[1]), dtype=torch.int32, device=logits.device),
                        torch.empty((len(idx),), dtype=torch.int32, device=logits.device)))
        io.append(row)
    return io


def move_some_full_kv_to_host(batches: List[Batch], on_host):
    """Like move_full_kv_to_host for the requests with on_host[j][i] true (batch j, request i);
    the others keep KV_full in HBM (None entries). Returns flat (host buffers, slots) lists over
    the batches' requests in order."""
    hs, ss = [], []
    for bt, flags in zip(batches, on_host):
        for b, (r, f) in enumerate(zip(bt.reqs, flags)):
            if not f:
                hs.append(None)
                ss.append(None)
                continue
            kv = torch.stack([r.k_full, r.v_full])
            h = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=True)
            h.copy_(kv)
            slot = torch.empty_like(kv)
            slot.copy_(kv)
            bt.set_full(b, slot[0], slot[1])
            hs.append(h)
            ss.append(slot)
            del kv
    torch.cuda.synchronize()
    return hs, ss


def move_full_kv_to_host(groups: List[Batch]):
    """After compression, move every request's KV_full to pinned host memory ([K; V] in one buffer
    per request) and give it a device staging slot of the same layout; the request's KV_full
    descriptor then points at the slot. Returns (host buffers, slots), per group and request."""
    host_kv, slots = [], []
    for bt in groups:
        hs, ss = [], []
        for b, r in enumerate(bt.reqs):
            kv = torch.stack([r.k_full, r.v_full])
            h = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=True)
            h.copy_(kv)
            slot = torch.empty_like(kv)
            bt.set_full(b, slot[0], slot[1])
            hs.append(h)
            ss.append(slot)
            del kv
        host_kv.append(hs)
        slots.append(ss)
    torch.cuda.synchronize()
    return host_kv, slots
