#!/usr/bin/env python
"""Benchmark of one VeriCache round on GB300: compress (keep-set) -> L draft steps -> verify -> accept.

Workload: Llama-3-8B attention shape, batch 8, 32/8 heads, d 128, context 32768, 4x token drop
(keep 8192 = last 512 + top 7680 by importance), L = 32 drafts, vocab 128256, planted match
probability 0.95; full KV resident in HBM (1.07 GB, larger than L2, so no flush is needed).
Metric: verified tokens/s = sum of accepted tokens (n_acc) over requests / round time, one
attention layer (no weights, MLP or LM head: an attention-only proxy).

  python bench.py [--gpus N --steps K --warmup W]      # the product path (CUDA kernels)
  python bench.py --impl reference ...                  # the CPU oracle on the host cores

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs its own replica of the
workload (the path has no exchange step): value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s/GPU (draft+verify+accept)"
UNIT = "tokens/s"
PROFILE = os.path.join(ROOT, "profiles", "draft_attn_llama8b_drop4x.md")
DRAFT_SOURCES = ["lossless_compressed_kv_vc_gb300/csrc/draft.cu", "lossless_compressed_kv_vc_gb300/csrc/vc_internal.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample-heads", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--child-steps", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--workload", default="llama8b_drop",
                    choices=["llama8b_drop", "qwen_quant2", "offload", "stagger", "importance"],
                    help="llama8b_drop: the headline round; qwen_quant2: the same round on the Qwen-32B-like "
                         "2-bit workload (16 x 65536 tokens, L 25); offload: Llama-70B-shape 4-bit requests with KV_full "
                         "in pinned host memory, two drafting while two stage and verify; stagger: the 16 "
                         "2-bit requests of the mixed serving workload (half with KV_full on the host) under "
                         "a naive split and under the planner's split; importance: SnapKV-style importance of the "
                         "headline workload's contexts from a 32-token observation window")
    ap.add_argument("--window", type=int, default=32, help="importance workload: observation window")
    ap.add_argument("--ctx-div", type=int, default=1,
                    help="offload workload: divide the context (a smaller case for profiler captures)")
    ap.add_argument("--compact", action="store_true",
                    help="gather the kept rows into a contiguous copy at compress time (inside the timed round)")
    ap.add_argument("--batch", type=int, default=None,
                    help="run only the first B requests (a smaller case for profiler captures)")
    ap.add_argument("--head-chunks", type=int, default=1,
                    help="offload workload: stage KV_full in this many KV-head ranges and verify each range as "
                         "soon as it lands (1 = stage the whole group, then verify)")
    ap.add_argument("--draft-steps", type=int, default=None,
                    help="offload and stagger workloads: drafts per round for every request (default: the "
                         "workload's L)")
    a = ap.parse_args()
    global _BATCH, _WORKLOAD
    _BATCH = a.batch
    _WORKLOAD = a.workload
    return a


_BATCH = None
_WORKLOAD = "llama8b_drop"


def workload():
    from workloads import configs
    w = configs.qwen32b_quant2() if _WORKLOAD == "qwen_quant2" else configs.llama8b_drop()
    if _BATCH is not None and _BATCH < w.B:
        w = configs.scaled(w, batch=_BATCH)
    return w


# ------------------------------------------------------------------------------------------------
# CPU oracle leg (reference arm and cpu_baseline): one request's round on a sample of KV heads
# ------------------------------------------------------------------------------------------------
def oracle_inputs(w, b: int):
    """Request b's round inputs as float32 numpy arrays (generated once per child process)."""
    import torch
    from workloads import gen
    ri = gen.request(w, 0, b, "cpu")
    draft, logits, L = gen.drafts_and_logits(w, 0, "cpu")
    f = lambda t: t.to(torch.float32).numpy()
    return (f(ri.k_full), f(ri.v_full), f(ri.q), f(ri.k_new), f(ri.v_new), ri.importance.numpy(),
            logits[b].numpy(), draft[b].numpy())


def oracle_round_sample(w, b: int, n_heads: int, inputs=None):
    """Time the oracle on request b: keep-set, L draft steps and verify for `n_heads` KV heads,
    accept. Returns (seconds scaled to all KV heads of the request, n_acc)."""
    import numpy as np
    import oracle as O
    kf, vf, q, kn, vn, imp, lg, dr = inputs if inputs is not None else oracle_inputs(w, b)
    G = w.Hq // w.Hkv
    t0 = time.perf_counter()
    idx = O.keep_set(imp, w.keep[b], w.recent[b])
    t_keep = time.perf_counter() - t0
    t1 = time.perf_counter()
    for hk in range(n_heads):
        sel = slice(hk * G, (hk + 1) * G)
        km, vm = kf[hk:hk + 1, idx], vf[hk:hk + 1, idx]
        empty = np.zeros((1, 0, w.d), np.float32)
        O.draft_round(q[:, sel], km, vm, empty, empty, kn[:, hk:hk + 1], vn[:, hk:hk + 1])
        O.verify_attn(q[:, sel], kf[hk:hk + 1], vf[hk:hk + 1], kn[:, hk:hk + 1].transpose(1, 0, 2),
                      vn[:, hk:hk + 1].transpose(1, 0, 2))
    t_heads = time.perf_counter() - t1
    t2 = time.perf_counter()
    _, n_acc = O.accept(lg, dr, w.L[b])
    t_acc = time.perf_counter() - t2
    return t_keep + t_heads * (w.Hkv / n_heads) + t_acc, n_acc


def cpu_child(args):
    """Runs in a fresh single-threaded process (BLAS threads pinned to 1 by the parent): oracle
    samples of request (i mod B) for i < child_steps, each on `sample_heads` KV heads; prints one
    JSON list of {secs_per_request, n_acc}."""
    w = workload()
    out, cache = [], {}
    for i in range(args.child_steps):
        b = i % w.B
        if b not in cache:
            cache[b] = oracle_inputs(w, b)
        secs, n_acc = oracle_round_sample(w, b, args.sample_heads, cache[b])
        out.append({"secs_per_request": secs, "n_acc": n_acc})
    print(json.dumps(out))


def run_cpu_child(sample_heads=1, steps=1):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", "--sample-heads",
                          str(sample_heads), "--child-steps", str(steps)], capture_output=True, text=True, env=env,
                         cwd=ROOT)
    wall = time.perf_counter() - t0
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1]), wall


def cpu_baseline_obj(w, rs):
    """The oracle over one whole round: every request, every KV head (no scaling)."""
    secs = sum(r["secs_per_request"] for r in rs)
    n_acc = sum(r["n_acc"] for r in rs)
    return {"value": n_acc / secs, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu_s": secs,
            "sample": f"one whole round of {w.name}: {w.B} requests x {w.Hkv} KV heads, keep-set, {w.L[0]} draft "
                      f"steps, verify and accept; numpy float64, one thread"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload()
    # one single-threaded child runs every step: step i samples request (i mod B) on one KV head
    # (time x Hkv), so a step is ~0.1 s of oracle work and the whole run a few minutes at most
    rs, _ = run_cpu_child(1, args.warmup + args.steps)
    timed = rs[args.warmup:]
    t = statistics.mean(r["secs_per_request"] for r in timed)
    value = sum(r["n_acc"] for r in timed) / sum(r["secs_per_request"] for r in timed)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3 * w.B,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"per step: request (step mod {w.B}) of {w.name}, 1 of {w.Hkv} KV heads "
                                       f"timed, x{w.Hkv}; ms_per_step is per round of {w.B} requests"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# native leg
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                out, _ = self.p.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def draft_source_hash():
    h = hashlib.sha256()
    for f in DRAFT_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the draft kernel from the committed ncu summary, or None when the
    kernel source changed since it was taken."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch\s*=\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256_16\s*=\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != draft_source_hash():
        return None
    return float(m.group(1))


def draft_algorithmic_bytes(w):
    """Bytes one draft step must move, summed over requests, averaged over the L steps: the kept
    K and V rows (keep x Hkv x 2 x d x 2 B), the window rows read, the index list (once per
    request), q in and o out, and the new row read and stored."""
    from workloads import DROP
    d, total = w.d, 0.0
    for b in range(w.B):
        win_avg = (w.L[b] + 1) / 2.0  # window rows 1..L over the round
        if w.mode[b] == DROP:
            keep = min(w.keep[b], w.ctx[b])
            total += w.Hkv * (keep + win_avg) * 2 * d * 2
            total += keep * 4
        else:  # quantised groups: codes, fp16 scales and zeros; then the bf16 residual and window
            ng = max(0, (w.ctx[b] - w.residual_min) // 32)
            total += w.Hkv * 32 * ng * (2 * d * w.bits // 8 + 2 * 4 * d // 32)
            total += w.Hkv * (w.ctx[b] - 32 * ng + win_avg) * 2 * d * 2
        total += 2 * w.Hq * d * 2
        total += 2 * 2 * w.Hkv * d * 2
    return total


def setup_native(w, device, compact=False):
    import torch
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import engine, VC_TOKEN_DROP, VC_QUANT
    from workloads import gen, DROP
    reqs = []
    for b in range(w.B):
        ri = gen.request(w, 0, b, device)
        reqs.append(engine.Req(mode=VC_TOKEN_DROP if w.mode[b] == DROP else VC_QUANT, ctx=w.ctx[b], L=w.L[b],
                               k_full=ri.k_full, v_full=ri.v_full, q=ri.q, k_new=ri.k_new, v_new=ri.v_new,
                               importance=ri.importance, keep=w.keep[b], recent=w.recent[b], compact=compact,
                               bits=w.bits))
    bt = engine.Batch(w.Hq, w.Hkv, w.d, reqs, residual_min=w.residual_min, device=device)
    bt.compress()
    bt.prepare_steps()
    draft, logits, L = gen.drafts_and_logits(w, 0, device)
    out_tokens = torch.empty((w.B, w.L_max + 1), dtype=torch.int32, device=device)
    n_acc = torch.empty((w.B,), dtype=torch.int32, device=device)
    return bt, draft, logits, L, out_tokens, n_acc


def aggregate(t_ms: float, tokens: int, dist=None, device="cpu"):
    """Whole-job figures over ranks: (the slowest rank's time in ms, the tokens of all ranks). Each
    rank passes its own time and token count; without a process group the local figures return."""
    if dist is None:
        return t_ms, tokens
    import torch
    t = torch.tensor([t_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(round(n.item()))


def run_native(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    w = workload()
    bt, draft, logits, L, out_tokens, n_acc = setup_native(w, device, compact=args.compact)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        bt.run_round(logits, draft, L, out_tokens, n_acc, stream)
    barrier()
    assert int(bt.dev_status.item()) == 0, "device status set during warm-up"
    tokens_per_step = int(n_acc.sum().item())

    # timed region: K rounds, inputs resident in HBM
    # one event pair around the draft phase (all L draft launches) of every timed round, on the
    # kernels' stream; events between single launches would hold back each step's early start
    ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        e0.record(stream)
        for k in range(args.steps):
            bt.run_round(logits, draft, L, out_tokens, n_acc, stream, draft_events=ev[k])
        e1.record(stream)
        barrier()
    draft_ms = [a.elapsed_time(b) / w.L_max for a, b in ev]  # per draft step (one vc_draft_attn call)
    t_ms = e0.elapsed_time(e1)
    t_max, tokens_all = aggregate(t_ms, tokens_per_step * args.steps, dist, device)
    assert int(bt.dev_status.item()) == 0, "device status set during the timed region"
    ms_per_step = t_max / args.steps
    value = tokens_all / (t_max / 1e3)

    # end-to-end through the public API with host buffers: H2D of the round's inputs, round, D2H
    e2e = run_e2e(w, bt, draft, logits, L, out_tokens, n_acc, stream, args.e2e_steps or max(3, min(args.steps, 100)),
                  barrier, dist, world, device)

    peaks, peak_kind = measured_peaks()
    from workloads import DROP
    quant = 0 if w.mode[0] == DROP else 1
    alg = draft_algorithmic_bytes(w)
    d_ms = statistics.mean(draft_ms)
    achieved = alg / (d_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": achieved / float(peaks["hbm_gbs"]), "traffic": profiled_traffic(),
                "kernel": "draft_attn_kernel<128,%d,1> (one vc_draft_attn call, partial merge included; mean over "
                          "the draft phase of each timed round)" % (0 if quant == 0 else w.bits),
                "algorithmic_bytes_per_launch": alg, "avg_launch_ms": d_ms, "peak_kind": peak_kind}
    # keep-set (+ gather when compacting), one draft launch per step, verify + its merge, accept (2)
    launches_per_step = (3 if quant else 1) + (1 if args.compact else 0) + w.L_max + 2 + 2
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "compact_keep_set": bool(args.compact), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "ctx": w.ctx[0],
                       "keep": w.keep[0], "recent": w.recent[0], "L": w.L[0], "V": w.V, "p": w.p[0],
                       "tokens_per_step": tokens_per_step,
                       "l2": "inputs larger than L2 (full KV 1.07 GB, kept rows 268 MB per draft step, logits 135 MB)"
                       if not quant else "inputs larger than L2 (full KV 4.3 GB, quantised cache 812 MB per draft "
                                         "step, logits 243 MB)"},
            "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "roofline": roofline,
            "clocks": clk.summary()}
    if quant:
        line["config"].update({"bits": w.bits, "keep": None, "recent": None})
        line["roofline"]["traffic"] = None
    if rank == 0 and not args.no_cpu_baseline and not quant:
        rs, wall = run_cpu_child(w.Hkv, w.B)
        cb = cpu_baseline_obj(w, rs)
        cb["wall_s"] = wall
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_e2e(w, bt, draft, logits, L, out_tokens, n_acc, stream, steps, barrier, dist, world, device):
    """Each step is one call of the engine's host-input round: that round's inputs (queries,
    drafted K/V, importance, drafts, logits, L) are copied from pinned host memory, the round runs
    through the C ABI, and n_acc and the accepted tokens are read back into pinned host memory.
    The accept inputs cross the host link on a second stream while the GPU drafts."""
    import torch
    from lossless_compressed_kv_vc_gb300 import engine
    hr = engine.HostRound(bt, logits, draft, L, out_tokens, n_acc)
    copy_stream = torch.cuda.Stream()
    h2d, d2h = hr.h2d_bytes, hr.d2h_bytes

    def step():
        bt.run_round_from_host(hr, stream, copy_stream)

    step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    t, tokens = aggregate(e0.elapsed_time(e1), int(hr.host_n_acc.sum().item()) * steps, dist, device)
    return {"value": tokens / (t / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps}


def run_offload(args):
    """Staggered offload periods: group A drafts while group B's KV_full is staged, B verifies and
    accepts; then the roles swap. value = accepted tokens of the four requests per period / period."""
    import torch
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import engine, VC_QUANT, vc_stage_full_kv
    from workloads import configs, gen
    w = configs.llama70b_offload4()
    if args.ctx_div > 1 or args.draft_steps is not None:
        w = configs.scaled(w, ctx_div=args.ctx_div, L=args.draft_steps)
    device = "cuda"
    groups = []
    for grp in ([0, 1], [2, 3]):
        rs = []
        for b in grp:
            ri = gen.request(w, 0, b, device)
            rs.append(engine.Req(mode=VC_QUANT, ctx=w.ctx[b], L=w.L[b], k_full=ri.k_full, v_full=ri.v_full, q=ri.q,
                                 k_new=ri.k_new, v_new=ri.v_new, bits=w.bits))
        bt = engine.Batch(w.Hq, w.Hkv, w.d, rs, residual_min=w.residual_min, device=device)
        bt.compress()
        groups.append(bt)
    host_kv, slots = engine.move_full_kv_to_host(groups)
    for bt in groups:
        bt.prepare_steps()
    draft, logits, L = gen.drafts_and_logits(w, 0, device)
    io = []
    for gi in range(2):
        sl = slice(2 * gi, 2 * gi + 2)
        io.append((logits[sl].contiguous(), draft[sl].contiguous(), L[sl].contiguous(),
                   torch.empty((2, w.L_max + 1), dtype=torch.int32, device=device),
                   torch.empty((2,), dtype=torch.int32, device=device)))
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    sg = engine.StaggeredOffload(groups, host_kv, slots, cs, ks, head_chunks=args.head_chunks)
    mk = lambda: [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    stage_bytes = sum(h.numel() * h.element_size() for h in host_kv[0])
    # host link alone: one group's KV_full, nothing else running
    alone = []
    for _ in range(3):
        e = mk()
        torch.cuda.synchronize()
        e[0].record(cs)
        for h, d in zip(host_kv[0], slots[0]):
            vc_stage_full_kv(h, d, h.numel() * h.element_size(), 64 << 20, cs, None)
        e[1].record(cs)
        torch.cuda.synchronize()
        alone.append(e[0].elapsed_time(e[1]))
    link_alone = stage_bytes / (min(alone) / 1e3) / 1e9
    for _ in range(args.warmup):
        sg.period(io)
    torch.cuda.synchronize()
    evs = [{k: mk() for k in ("draft0", "draft1", "stage0", "stage1")} for _ in range(args.steps)]
    for ev in evs:
        ev["verified0"], ev["verified1"] = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0, e1 = mk()
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        e0.record(ks)
        for k in range(args.steps):
            sg.period(io, evs[k])
        e1.record(ks)
        torch.cuda.synchronize()
    t_ms = e0.elapsed_time(e1)
    for bt in groups:
        assert int(bt.dev_status.item()) == 0
    tokens = int(io[0][4].sum().item() + io[1][4].sum().item())
    # overlap: how much of each copy interval lies inside some draft interval (the copy stream runs
    # ahead of the compute stream, so a copy may land under either phase's drafting)
    copy_iv, draft_iv = [], []
    for ev in evs:
        for dk in ("draft0", "draft1"):
            draft_iv.append((e0.elapsed_time(ev[dk][0]), e0.elapsed_time(ev[dk][1])))
        for sk in ("stage0", "stage1"):
            copy_iv.append((e0.elapsed_time(ev[sk][0]), e0.elapsed_time(ev[sk][1])))
    # verification left once a group's copy has landed and the other group's drafting is done (the
    # verify of a group follows the drafting phase on the compute stream)
    exposed = []
    for ev in evs:
        for g_ver, dk in ((1, "draft0"), (0, "draft1")):
            ready = max(e0.elapsed_time(ev["stage%d" % g_ver][1]), e0.elapsed_time(ev[dk][1]))
            exposed.append(e0.elapsed_time(ev["verified%d" % g_ver]) - ready)
    copy_ms = [b - a for a, b in copy_iv]
    draft_ms = [b - a for a, b in draft_iv]
    overlap = [sum(max(0.0, min(b, d1) - max(a, d0)) for d0, d1 in draft_iv) / max(1e-9, b - a) for a, b in copy_iv]
    link_loaded = stage_bytes / (statistics.mean(copy_ms) / 1e3) / 1e9
    peaks, peak_kind = measured_peaks()
    G = w.Hq // w.Hkv
    ng = (w.ctx[0] - w.residual_min) // 32
    per_req = w.Hkv * (32 * ng * (2 * w.d * w.bits // 8 + 2 * 4 * w.d // 32) + (w.ctx[0] - 32 * ng + (w.L[0] + 1) / 2) * 2 * w.d * 2)
    alg = 2 * per_req + 2 * (2 * w.Hq * w.d * 2 + 4 * w.Hkv * w.d * 2)
    step_ms = statistics.mean(draft_ms) / w.L[0]
    achieved = alg / (step_ms / 1e3) / 1e9
    line = {"metric": METRIC, "value": tokens * args.steps / (t_ms / 1e3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "ctx": w.ctx[0],
                       "bits": w.bits, "L": w.L[0], "V": w.V, "tokens_per_period": tokens,
                       "step": "one period: each of the 4 requests drafts L steps and is staged, verified and accepted once"},
            "stage": {"bytes_per_copy": stage_bytes, "link_alone_gbs": link_alone, "link_during_draft_gbs": link_loaded,
                      "frac_of_link": link_loaded / link_alone, "copy_ms": statistics.mean(copy_ms),
                      "draft_phase_ms": statistics.mean(draft_ms), "copy_overlapped_by_draft": statistics.mean(overlap),
                      "head_chunks": args.head_chunks, "verify_after_copy_and_draft_ms": statistics.mean(exposed)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": achieved / float(peaks["hbm_gbs"]), "traffic": None,
                         "kernel": "draft_attn_kernel<128,4> (2 requests per call), mean over a draft phase",
                         "algorithmic_bytes_per_launch": alg, "avg_launch_ms": step_ms, "peak_kind": peak_kind},
            "clocks": clk.summary()}
    print(json.dumps(line))
    return 0


def run_stagger(args):
    """The quantised requests of the mixed serving workload (contexts log-uniform 8K-256K, L 25-40,
    KV_full of half of them in pinned host memory) staggered in two groups. Per-request costs come
    from rates measured on the workload itself (the whole batch's draft phase and verification,
    one request's copy alone) times each request's bytes; the period is then measured for a naive
    split (first half / second half), an alternating split and the planner's split."""
    import torch
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import (engine, VC_QUANT, vc_draft_attn, vc_verify_attn, vc_stage_full_kv,
                                                 vc_stagger_period)
    from workloads import configs, gen
    full = configs.mixed_serving()
    w = configs.subset(full, full.request_indices("quant"), name="mixed_quant2_stagger_16req_ctx8k_256k")
    if args.ctx_div > 1 or args.draft_steps is not None:
        w = configs.scaled(w, ctx_div=args.ctx_div, L=args.draft_steps)
    dev = "cuda"
    reqs, host, slot = [], [], []
    for b in range(w.B):
        ri = gen.request(w, 0, b, dev)
        kf, vf = ri.k_full, ri.v_full
        h = s = None
        if w.on_host[b]:
            s = torch.stack([kf, vf])  # device staging slot; the request's KV_full descriptor points at it
            h = torch.empty(s.shape, dtype=s.dtype, pin_memory=True)
            h.copy_(s)
            kf, vf = s[0], s[1]
        host.append(h)
        slot.append(s)
        reqs.append(engine.Req(mode=VC_QUANT, ctx=w.ctx[b], L=w.L[b], k_full=kf, v_full=vf, q=ri.q, k_new=ri.k_new,
                               v_new=ri.v_new, bits=w.bits))
    del ri
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def timed(fn, stream, reps=3):
        best = float("inf")
        for _ in range(reps + 1):
            e = mk()
            torch.cuda.synchronize()
            e[0].record(stream)
            fn()
            e[1].record(stream)
            torch.cuda.synchronize()
            best = min(best, e[0].elapsed_time(e[1]))
        return best * 1e6  # ns

    # rates measured on the whole batch
    cal = engine.Batch(w.Hq, w.Hkv, w.d, reqs, residual_min=w.residual_min, device=dev)
    cal.compress()
    cal.prepare_steps()
    t_draft = timed(lambda: [vc_draft_attn(sh, arr, cal.ws_draft, cal.dev_status, ks) for sh, arr, act in cal._steps], ks)
    t_verify = timed(lambda: vc_verify_attn(cal.shape, cal._verify_arr, cal.ws_verify, cal.dev_status, ks), ks)
    assert int(cal.dev_status.item()) == 0
    del cal
    d, b8 = w.d, w.bits
    ng = [max(0, (c - w.residual_min) // 32) for c in w.ctx]
    step_bytes = [w.Hkv * (32 * n * (2 * d * b8 // 8 + 2 * 4 * d // 32) + (c - 32 * n + (L + 1) / 2) * 2 * d * 2)
                  for n, c, L in zip(ng, w.ctx, w.L)]
    draft_bytes = [L * sb for L, sb in zip(w.L, step_bytes)]
    verify_bytes = [w.Hkv * (c + L) * 2 * d * 2 + (L + 1) * w.V * 4 for c, L in zip(w.ctx, w.L)]
    full_bytes = [2 * w.Hkv * c * d * 2 for c in w.ctx]
    hb = next(b for b in range(w.B) if w.on_host[b])
    t_link = timed(lambda: vc_stage_full_kv(host[hb], slot[hb], full_bytes[hb], 64 << 20, cs, None), cs)
    rate_d, rate_v = sum(draft_bytes) / t_draft, sum(verify_bytes) / t_verify
    rate_s = full_bytes[hb] / t_link
    costs = engine.stagger_costs([x / rate_d for x in draft_bytes], [x / rate_v for x in verify_bytes],
                                 [fb / rate_s if w.on_host[b] else 0 for b, fb in enumerate(full_bytes)])
    g0, g1, t_plan = engine.plan_groups(costs)
    half = w.B // 2
    splits = {"halves": [0] * half + [1] * (w.B - half), "alternate": [b % 2 for b in range(w.B)],
              "planned": [0 if b in g0 else 1 for b in range(w.B)]}
    draft, logits, Lt = gen.drafts_and_logits(w, 0, dev)
    out = {}
    for name, grp in splits.items():
        idx = [[b for b in range(w.B) if grp[b] == gi] for gi in (0, 1)]
        if not idx[0] or not idx[1]:
            out[name] = {"skipped": "empty group"}
            continue
        groups, io = [], []
        for gi in (0, 1):
            bt = engine.Batch(w.Hq, w.Hkv, w.d, [reqs[b] for b in idx[gi]], residual_min=w.residual_min, device=dev)
            bt.compress()
            bt.prepare_steps()
            groups.append(bt)
            sel = torch.tensor(idx[gi], device=dev)
            n = len(idx[gi])
            io.append((logits[sel].contiguous(), draft[sel].contiguous(), Lt[sel].contiguous(),
                       torch.empty((n, w.L_max + 1), dtype=torch.int32, device=dev),
                       torch.empty((n,), dtype=torch.int32, device=dev)))
        sg = engine.StaggeredOffload(groups, [[host[b] for b in idx[gi]] for gi in (0, 1)],
                                     [[slot[b] for b in idx[gi]] for gi in (0, 1)], cs, ks)
        for _ in range(args.warmup):
            sg.period(io)
        torch.cuda.synchronize()
        e = mk()
        e[0].record(ks)
        for _ in range(args.steps):
            sg.period(io)
        e[1].record(ks)
        torch.cuda.synchronize()
        for bt in groups:
            assert int(bt.dev_status.item()) == 0
        t_ms = e[0].elapsed_time(e[1])
        tokens = int(io[0][4].sum().item() + io[1][4].sum().item())
        out[name] = {"groups": grp, "period_ms": t_ms / args.steps, "modelled_ms": vc_stagger_period(costs, grp)[1] / 1e6,
                     "tokens_per_s": tokens * args.steps / (t_ms / 1e3)}
        del groups, io, sg
    best_naive = max(v.get("tokens_per_s", 0.0) for k, v in out.items() if k != "planned")
    line = {"metric": METRIC, "value": out["planned"]["tokens_per_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": out["planned"]["period_ms"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "ctx": w.ctx, "L": w.L,
                       "bits": w.bits, "on_host": w.on_host,
                       "step": "one period: every request drafts its L steps, is staged if its KV_full is on the "
                               "host, verified and accepted once"},
            "stagger": {"rates_gbs": {"draft": rate_d, "verify": rate_v, "link": rate_s},
                        "costs_ns": costs, "planned_period_ms": t_plan / 1e6, "splits": out,
                        "planned_over_best_naive": out["planned"]["tokens_per_s"] / best_naive if best_naive else None}}
    print(json.dumps(line))
    return 0


def run_importance(args):
    """SnapKV-style importance (vc_snapkv_importance, 4 launches) for every request of the headline
    workload (8 x 32768 context tokens, 32/8 heads, d 128), window 32, max pooling of width 7.
    value = context tokens scored per second. Roofline: the two passes read every key twice
    (2 x Hkv x ctx x d x 2 B per request) and do 2 x 2 x (W G) x ctx x d x Hkv flops."""
    import torch
    from workloads import gen
    w = workload()
    device = "cuda"
    bt, *_ = setup_native(w, device)
    q_obs = [gen.observation_queries(w, b, args.window, device) for b in range(w.B)]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        bt.snapkv_importance(q_obs, args.window, 7, stream=stream)
    torch.cuda.synchronize()
    assert int(bt.dev_status.item()) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            bt.snapkv_importance(q_obs, args.window, 7, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
    t_ms = e0.elapsed_time(e1) / args.steps
    G, R = w.Hq // w.Hkv, args.window * w.Hq // w.Hkv
    tokens = sum(w.ctx)
    key_bytes = sum(2 * w.Hkv * c * w.d * 2 for c in w.ctx)
    flops = sum(2 * 2 * R * c * w.d * w.Hkv for c in w.ctx)
    peaks, kind = measured_peaks()
    gbs, tfs = key_bytes / (t_ms / 1e3) / 1e9, flops / (t_ms / 1e3) / 1e12
    line = {"metric": "SnapKV-style importance: context tokens scored/s", "value": tokens / (t_ms / 1e3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name + "_importance", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                       "ctx": w.ctx[0], "window": args.window, "rows_per_kv_head": R, "pool": "max 7",
                       "l2": "keys 1.07 GB per pass, larger than L2"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                         "tensor_tflops": tfs, "tensor_frac_of_bf16_peak": tfs / float(peaks["bf16_tflops"]),
                         "kernel": "imp_stats + imp_lse + imp_votes + imp_pool (one vc_snapkv_importance call)",
                         "algorithmic_bytes_per_launch": key_bytes, "flops_per_launch": flops, "peak_kind": kind},
            "clocks": clk.summary()}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.cpu_child:
        return cpu_child(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "offload":
        return run_offload(args)
    if args.workload == "stagger":
        return run_stagger(args)
    if args.workload == "importance":
        return run_importance(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main() or 0)
