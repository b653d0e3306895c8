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
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s/GPU (draft+verify+accept)"
UNIT = "tokens/s"
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
DRAFT_SOURCES = ["lossless_compressed_kv_vc_gb300/csrc/draft.cu", "lossless_compressed_kv_vc_gb300/csrc/draft_common.cuh",
                 "lossless_compressed_kv_vc_gb300/csrc/vc_internal.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 300 for this implementation; 20 for --impl reference, whose "
                         "steps are one request's whole round on the host cores each)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="mixed",
                    choices=["mixed", "llama8b_drop", "qwen_quant2", "offload", "stagger", "importance"],
                    help="mixed (default): the mixed staggered serving batch, 32 requests of 8K-256K tokens, half "
                         "token drop and half 2-bit, half with KV_full in pinned host memory, two groups planned by "
                         "the staggering planner; llama8b_drop: the Llama-3-8B-shape drop-4x round; "
                         "qwen_quant2: the same round on the Qwen-32B-like "
                         "2-bit workload (16 x 65536 tokens, L 25); offload: Llama-70B-shape 4-bit requests with KV_full "
                         "in pinned host memory, two drafting while two stage and verify; stagger: the 16 "
                         "2-bit requests of the mixed serving workload (half with KV_full on the host) under "
                         "a naive split and under the planner's split; importance: SnapKV-style importance of the "
                         "headline workload's contexts from a 32-token observation window")
    ap.add_argument("--window", type=int, default=32, help="importance workload: observation window")
    ap.add_argument("--no-graphs", action="store_true",
                    help="mixed workload: issue every draft call from the host instead of replaying each batch's "
                         "draft series as a captured CUDA graph")
    ap.add_argument("--timeline", default=None,
                    help="mixed workload: write every timed period's CUDA-event intervals (draft calls, verification, "
                         "staging copies; ms from the start of the timed region) and the host's issue times to this "
                         "JSON file")
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
    if a.steps is None:
        a.steps = 20 if a.impl == "reference" else 300
    global _BATCH, _WORKLOAD
    _BATCH = a.batch
    _WORKLOAD = a.workload
    return a


_BATCH = None
_WORKLOAD = "mixed"


def workload():
    from workloads import configs
    if _WORKLOAD == "mixed":
        w = configs.mixed_serving()
    else:
        w = configs.qwen32b_quant2() if _WORKLOAD == "qwen_quant2" else configs.llama8b_drop()
    if _BATCH is not None and _BATCH < w.B:
        w = configs.scaled(w, batch=_BATCH)
    return w


# ------------------------------------------------------------------------------------------------
# CPU oracle legs (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------------------
# The oracle runs on the host cores as a fixed pool of worker processes (spawn context: the parent
# may hold a CUDA context). One "wave" is one request of the workload: its query heads are split
# evenly over the workers (consecutive heads, so a worker's heads share KV heads), every worker
# prepares its inputs, all meet at a barrier, the parent starts its clock, the workers run the
# oracle's round for their heads (all draft steps, verification, and -- worker 0 -- accept), all meet
# at a second barrier and the clock stops. So a wave's time is the measured wall time of the
# round's arithmetic on all workers at once. Preparation (input generation, the keep-set and the
# quantisation of KV_comp, which the GPU round also does once per request, outside the round) is
# outside the clock. The credited tokens of a wave are the request's accepted tokens.

def _oracle_worker(wid, nworkers, task_q, result_q, barrier):
    import os as _os
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ[k] = "1"
    import numpy as np
    import torch
    torch.set_num_threads(1)
    import oracle as O
    from workloads import gen, DROP
    while True:
        task = task_q.get()
        if task is None:
            return
        w, b = task
        err, secs, n_acc = None, 0.0, 0
        try:
            G = w.Hq // w.Hkv
            h0, h1 = wid * w.Hq // nworkers, (wid + 1) * w.Hq // nworkers
            f = lambda t: t.to(torch.float32).numpy()
            k, v = gen.full_kv(w, b)
            q, kn, vn = gen.round_queries(w, 0, b)
            q, kn, vn = f(q), f(kn), f(vn)
            prep = []
            for j in sorted({h // G for h in range(h0, h1)}):
                kf, vf = f(k[j:j + 1]), f(v[j:j + 1])
                if w.mode[b] == DROP:
                    idx = O.keep_set(gen.importance(w, b).numpy(), w.keep[b], w.recent[b])
                    km, vm = O.comp_main_rows("drop", kf, vf, idx=idx)
                    kw0 = vw0 = np.zeros((1, 0, w.d), np.float32)
                else:
                    qkv = O.quantize_kv(kf, vf, w.bits, w.residual_min)
                    km, vm = O.comp_main_rows("quant", kf, vf, qkv=qkv)
                    kw0, vw0 = qkv["k_res"], qkv["v_res"]
                sel = [h for h in range(h0, h1) if h // G == j]
                prep.append((sel, kf, vf, km, vm, kw0, vw0, kn[:, j:j + 1], vn[:, j:j + 1]))
            del k, v
            dr, lg = gen.request_logits(w, 0, b) if wid == 0 else (None, None)
        except Exception as e:  # still meet the barriers, report the error
            err, prep = repr(e), []
        barrier.wait()
        t0 = time.perf_counter()
        try:
            for sel, kf, vf, km, vm, kw0, vw0, knj, vnj in prep:
                qs = q[:, sel]
                O.draft_round(qs, km, vm, kw0, vw0, knj, vnj)
                O.verify_attn(qs, kf, vf, knj.transpose(1, 0, 2), vnj.transpose(1, 0, 2))
            if wid == 0 and err is None:
                n_acc = O.accept(lg.numpy(), dr.numpy(), w.L[b])[1]
        except Exception as e:
            err = repr(e)
        secs = time.perf_counter() - t0
        barrier.wait()
        result_q.put((wid, err, secs, n_acc))


class OraclePool:
    """Worker processes that run the oracle's round of one request per wave (see above)."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n = workers or (os.cpu_count() or 1)
        self.barrier = ctx.Barrier(self.n + 1)
        self.result_q = ctx.Queue()
        self.task_q = [ctx.Queue() for _ in range(self.n)]
        env_keep = {k: os.environ.get(k) for k in ("CUDA_VISIBLE_DEVICES",)}
        os.environ["CUDA_VISIBLE_DEVICES"] = ""  # the workers never touch a GPU
        try:
            self.procs = [ctx.Process(target=_oracle_worker, args=(i, self.n, self.task_q[i], self.result_q,
                                                                   self.barrier), daemon=True)
                          for i in range(self.n)]
            for p in self.procs:
                p.start()
        finally:
            for k, v in env_keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def wave(self, w, b, timeout=1800):
        """Run request b's round on all workers; returns (wall seconds of the compute, summed
        worker seconds, accepted tokens)."""
        for q in self.task_q:
            q.put((w, b))
        self.barrier.wait(timeout)
        t0 = time.perf_counter()
        self.barrier.wait(timeout)
        wall = time.perf_counter() - t0
        res = [self.result_q.get(timeout=timeout) for _ in range(self.n)]
        errs = [e for _, e, _, _ in res if e]
        if errs:
            raise RuntimeError("oracle worker failed: " + errs[0])
        return wall, sum(r[2] for r in res), sum(r[3] for r in res)

    def close(self):
        for q in self.task_q:
            q.put(None)
        for p in self.procs:
            p.join(timeout=30)


def sample_requests(w, per_mode=1):
    """Requests of each compression mode whose contexts are nearest the mode's median (the
    cpu_baseline's bounded sample)."""
    import numpy as np
    out = []
    for m in sorted(set(w.mode)):
        idx = [b for b in range(w.B) if w.mode[b] == m]
        med = float(np.median([w.ctx[b] for b in idx]))
        out += sorted(idx, key=lambda b: (abs(w.ctx[b] - med), b))[:per_mode]
    return sorted(out)


def cpu_baseline_oracle(w):
    """The oracle on all host cores over a bounded sample: one round of each sampled request."""
    pool = OraclePool()
    try:
        reqs = sample_requests(w)
        walls, cpu, tok = 0.0, 0.0, 0
        for b in reqs:
            wall, c, n = pool.wave(w, b)
            walls, cpu, tok = walls + wall, cpu + c, tok + n
    finally:
        pool.close()
    return {"value": tok / walls, "unit": UNIT, "cores": pool.n, "host_cores": os.cpu_count(), "kind": "oracle",
            "single_thread_value": tok / cpu, "wall_s": walls, "cpu_s": cpu,
            "sample": "one round (all draft steps, verification and accept, every query head) of requests %s of %s "
                      "(the requests of each compression mode whose contexts are nearest the mode's median: %s "
                      "tokens), split over %d worker processes of one thread each; value = their accepted tokens / "
                      "the measured wall time of the arithmetic (KV_comp built beforehand, as on the GPU); "
                      "single_thread_value = the same tokens / the workers' summed seconds"
                      % (reqs, w.name, [w.ctx[b] for b in reqs], pool.n)}


def run_reference(args):
    """The oracle as the reference arm: one wave (one request's whole round on all host cores) per
    step, cycling through the workload's requests; value = accepted tokens of the timed waves / their
    measured wall time, ms_per_step = the mean wave wall time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload()
    order = list(range(w.B))
    pool = OraclePool()
    walls, toks, cpu = [], [], 0.0
    try:
        for i in range(args.warmup + args.steps):
            wall, c, n = pool.wave(w, order[i % w.B])
            if i >= args.warmup:
                walls.append(wall)
                toks.append(n)
                cpu += c
    finally:
        pool.close()
    value = sum(toks) / sum(walls)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(walls) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.n, "host_cores": os.cpu_count(),
                             "kind": "oracle", "single_thread_value": sum(toks) / cpu,
                             "sample": "per step: the whole round of one request of %s (requests in order, "
                                       "cycling), its query heads split over %d single-thread worker processes; "
                                       "the step time is the measured wall time of that arithmetic"
                                       % (w.name, pool.n)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# native leg
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs. Entering waits
    (up to 5 s) for the first sample, so that nvidia-smi's start-up (NVML initialisation, which can
    hold up GPU work for tens of ms) happens before the timed region; the summary uses the samples
    taken after that."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.p = None
        self.lines = []
        self._all = []

    def _read(self):
        for line in self.p.stdout:
            if line.strip():
                self._all.append(line)

    def __enter__(self):
        import threading
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self._all and time.time() - t0 < 5.0 and self.p.poll() is None:
            time.sleep(0.02)
        self._mark = len(self._all)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                self.p.wait()
            self._t.join(timeout=5)
            self.lines = self._all[self._mark:]

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


def profiled_traffic(kernel, workload_name):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of `kernel` on
    `workload_name` from profiles/traffic.json (written from an ncu capture), or None when there is
    no entry or the draft kernel's source changed since the capture."""
    try:
        entries = json.load(open(TRAFFIC))["entries"]
    except (OSError, ValueError, KeyError):
        return None
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload_name:
            return float(e["bytes_per_launch"]) if e.get("source_sha16") == draft_source_hash() else None
    return None


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
    from workloads import DROP
    quant = 0 if w.mode[0] == DROP else 1
    bt, draft, logits, L, out_tokens, n_acc = setup_native(w, device, compact=args.compact)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        bt.run_round(logits, draft, L, out_tokens, n_acc, stream, compress=not quant)
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
            bt.run_round(logits, draft, L, out_tokens, n_acc, stream, draft_events=ev[k], compress=not quant)
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
                  barrier, dist, world, device, quant)

    peaks, peak_kind = measured_peaks()
    alg = draft_algorithmic_bytes(w)
    d_ms = statistics.mean(draft_ms)
    achieved = alg / (d_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": achieved / float(peaks["hbm_gbs"]),
                "traffic": profiled_traffic("draft_attn_kernel<128,%d,1>" % (0 if quant == 0 else w.bits), w.name),
                "kernel": "draft_attn_kernel<128,%d,1> (one vc_draft_attn call, partial merge included; mean over "
                          "the draft phase of each timed round)" % (0 if quant == 0 else w.bits),
                "algorithmic_bytes_per_launch": alg, "avg_launch_ms": d_ms, "peak_kind": peak_kind}
    # keep-set (+ gather when compacting; quantised caches are built once, outside the round), one
    # draft launch per step, the verification's kernels and merges (as the library splits the
    # batch's KV heads), accept (2)
    launches_per_step = (0 if quant else 1) + (1 if args.compact else 0) + w.L_max + bt.verify_launches() + 2
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
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_oracle(w)
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------------------------
# mixed staggered serving batch (the default workload)
# ------------------------------------------------------------------------------------------------
def request_step_bytes(w, b, s, sz):
    """Algorithmic bytes of request b's draft step s: its KV_comp (kept K and V rows and the index
    list, or the quantised codes, fp16 scales and zeros), the window rows it reads (residual, the
    drafted rows so far and this step's own), q in, o out, and the new K/V row read and stored.
    sz: the request's vc_comp_bytes."""
    from workloads import DROP
    d, H = w.d, w.Hkv
    if w.mode[b] == DROP:
        main = H * sz.keep * 2 * d * 2 + sz.keep * 4
        win = s + 1
    else:
        ng = sz.ng
        main = H * 32 * ng * (2 * d * w.bits // 8) + H * ng * 2 * 2 * d + H * 32 * ng * 2 * 2 * (d // 32)
        win = sz.n_res + s + 1
    return main + H * win * 2 * d * 2 + 2 * w.Hq * d * 2 + 2 * 2 * H * d * 2


def request_verify_work(w, b):
    """(bytes, flops) of request b's verification: KV_full and the drafted rows read once per KV
    head, q in and o out; QK^T and PV over ctx + (i + 1) keys for draft row i."""
    d, H, G, L, ctx = w.d, w.Hkv, w.Hq // w.Hkv, w.L[b], w.ctx[b]
    byts = H * (ctx + L) * 2 * d * 2 + 2 * L * w.Hq * d * 2
    flops = 4 * d * G * H * (L * ctx + L * (L + 1) // 2)
    return byts, flops


def _covered(iv, cover):
    """Fraction of interval iv = (a, b) inside the union of the intervals `cover`."""
    a, b = iv
    pts = sorted((max(a, c0), min(b, c1)) for c0, c1 in cover if min(b, c1) > max(a, c0))
    tot, end = 0.0, a
    for c0, c1 in pts:
        if c1 > end:
            tot += c1 - max(c0, end)
            end = c1
    return tot / max(1e-12, b - a)


def run_mixed(args):
    """The mixed staggered serving batch: 32 requests, contexts log-uniform in 8K-256K, half token
    drop 4x (even requests) and half 2-bit (odd), KV_full of half of them in pinned host memory, L
    uniform in 25-40. KV_comp is built once per request (outside the timed region). A step is one
    period of cross-resource staggering over two groups chosen by the staggering planner from costs
    measured on the workload: group A drafts (one C-ABI call per compression mode per draft step)
    while group B's host-resident KV_full is staged over the host link, then B is verified and
    accepted; then the roles swap. Every request drafts its L steps, is staged if its KV_full is on
    the host, verified and accepted once per step."""
    import torch
    import __graft_entry__ as g
    g.build()
    from lossless_compressed_kv_vc_gb300 import (engine, VC_TOKEN_DROP, VC_QUANT, vc_draft_attn, vc_verify_attn,
                                                 vc_stage_full_kv, vc_comp_bytes, vc_shape, vc_stagger_period)
    from workloads import configs, gen, DROP
    w = configs.mixed_serving()
    if args.ctx_div > 1:
        w = configs.scaled(w, ctx_div=args.ctx_div)
    if args.batch is not None and args.batch < w.B:
        w = configs.subset(w, list(range(args.batch)))
    dev = "cuda"
    torch.cuda.set_device(0)
    B, d = w.B, w.d
    sizes = [vc_comp_bytes(vc_shape(1, w.Hq, w.Hkv, d), VC_TOKEN_DROP if w.mode[b] == DROP else VC_QUANT, w.bits,
                           w.ctx[b], w.ctx[b], w.keep[b], w.residual_min, w.L[b]) for b in range(B)]
    reqs = []
    for b in range(B):
        ri = gen.request(w, 0, b, dev)
        drop = w.mode[b] == DROP
        reqs.append(engine.Req(mode=VC_TOKEN_DROP if drop else VC_QUANT, ctx=w.ctx[b], L=w.L[b], k_full=ri.k_full,
                               v_full=ri.v_full, q=ri.q, k_new=ri.k_new, v_new=ri.v_new,
                               importance=ri.importance if drop else None, keep=w.keep[b], recent=w.recent[b],
                               compact=bool(drop and w.on_host[b]), bits=w.bits))
    del ri
    draft_b = [sum(request_step_bytes(w, b, s, sizes[b]) for s in range(w.L[b])) for b in range(B)]
    verify_b = [request_verify_work(w, b) for b in range(B)]
    full_b = [2 * w.Hkv * w.ctx[b] * d * 2 for b in range(B)]
    cs, ks = torch.cuda.Stream(), torch.cuda.Stream()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def timed(fn, stream, reps=2):
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

    # --- costs for the planner: rates measured on the workload itself (each mode's whole draft
    # phase, the whole verification, one host-resident request's copy alone) times each request's bytes
    modes = [m for m in (DROP, "quant") if m in w.mode]
    rate = {}
    ver_ns, ver_bytes = 0.0, 0
    for m in modes:
        idx = [b for b in range(B) if w.mode[b] == m]
        cal = engine.Batch(w.Hq, w.Hkv, d, [reqs[b] for b in idx], residual_min=w.residual_min, device=dev)
        cal.compress(ks)
        cal.prepare_steps()
        t = timed(lambda: [vc_draft_attn(sh, arr, cal.ws_draft, cal.dev_status, ks) for sh, arr, act in cal._steps], ks)
        rate[m] = sum(draft_b[b] for b in idx) / t
        ver_ns += timed(lambda: vc_verify_attn(cal.shape, cal._verify_arr, cal.ws_verify, cal.dev_status, ks), ks)
        ver_bytes += sum(verify_b[b][0] for b in idx)
        assert int(cal.dev_status.item()) == 0
        del cal
    rate_v = ver_bytes / ver_ns
    ver_alone = {"tflops": sum(verify_b[b][1] for b in range(B)) / ver_ns / 1e3, "gbs": rate_v,
                 "ms": ver_ns / 1e6}  # every request verified, one call per mode, nothing else running
    host_reqs = [b for b in range(B) if w.on_host[b]]
    rate_s, link_alone = None, None
    if host_reqs:
        hb = min(host_reqs, key=lambda b: abs(w.ctx[b] - sorted(w.ctx)[B // 2]))
        src = torch.empty((full_b[hb] // 2,), dtype=torch.bfloat16, pin_memory=True)
        dst = torch.empty((full_b[hb] // 2,), dtype=torch.bfloat16, device=dev)
        t = timed(lambda: vc_stage_full_kv(src, dst, full_b[hb], 64 << 20, cs, None), cs)
        rate_s = full_b[hb] / t
        link_alone = rate_s
        del src, dst
    costs = engine.stagger_costs([draft_b[b] / rate[w.mode[b]] for b in range(B)],
                                 [verify_b[b][0] / rate_v for b in range(B)],
                                 [full_b[b] / rate_s if w.on_host[b] else 0 for b in range(B)])
    g0, g1, t_plan = engine.plan_groups(costs)
    split = [0 if b in g0 else 1 for b in range(B)]

    # --- the two groups, one batch per compression mode in each; KV_comp built once
    draft, logits, Lt = gen.drafts_and_logits(w, 0, dev)
    groups, members, host_kv, slots = engine.staggered_groups(w.Hq, w.Hkv, d, reqs, split, w.on_host,
                                                              w.residual_min, dev, ks)
    io = engine.group_io(members, logits, draft, Lt)
    torch.cuda.synchronize()
    sg = engine.StaggeredOffload(groups, host_kv, slots, cs, ks, head_chunks=args.head_chunks)
    for k in range(args.warmup):
        sg.period(io)
        if k == 0 and not args.no_graphs:
            sg.capture_drafts()  # each batch's draft series as one CUDA graph (one host launch)
    torch.cuda.synchronize()
    for bts in groups:
        for bt in bts:
            assert int(bt.dev_status.item()) == 0, "device status set during warm-up"
    tokens = sum(int(t[4].sum().item()) for gi in (0, 1) for t in io[gi])

    evs = []
    for _ in range(args.steps):
        ev = {"draft%d" % gi: [mk() for _ in groups[gi]] for gi in (0, 1)}
        ev.update({k: mk() for k in ("stage0", "stage1", "verify0", "verify1")})
        evs.append(ev)
    e0, e1 = mk()
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        e0.record(ks)
        cs.wait_event(e0)
        h0 = time.perf_counter()
        host_t = []
        for k in range(args.steps):
            host_t.append((time.perf_counter() - h0) * 1e3)
            sg.period(io, evs[k])
        e1.record(ks)
        host_ms = (time.perf_counter() - h0) * 1e3  # the host's time to issue every call of the timed periods
        torch.cuda.synchronize()
    t_ms = e0.elapsed_time(e1)
    for bts in groups:
        for bt in bts:
            assert int(bt.dev_status.item()) == 0, "device status set during the timed region"
    value = tokens * args.steps / (t_ms / 1e3)

    # --- per-kernel time from the events (each interval on the stream that ran it)
    rel = lambda e: e0.elapsed_time(e)
    kind_ms = {m: 0.0 for m in modes}
    kind_launch = {m: 0 for m in modes}
    kind_bytes = {m: 0.0 for m in modes}
    comp_iv, copy_iv = [], []
    for ev in evs:
        for gi in (0, 1):
            for (a, b_), bt, idx in zip(ev["draft%d" % gi], groups[gi], members[gi]):
                m = w.mode[idx[0]]
                kind_ms[m] += a.elapsed_time(b_)
                kind_launch[m] += len(bt._steps)
                kind_bytes[m] += sum(draft_b[b] for b in idx)
                comp_iv.append((rel(a), rel(b_)))
            a, b_ = ev["verify%d" % gi]
            comp_iv.append((rel(a), rel(b_)))
            a, b_ = ev["stage%d" % gi]
            if sg.stage_bytes(gi):
                copy_iv.append((rel(a), rel(b_)))
    ver_ms = sum(ev["verify%d" % gi][0].elapsed_time(ev["verify%d" % gi][1]) for ev in evs for gi in (0, 1))
    stage_ms = sum(b_ - a for a, b_ in copy_iv)
    peaks, peak_kind = measured_peaks()
    hbm, bf16 = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops_sustained"])
    ver_bytes_p = sum(v[0] for v in verify_b)
    ver_flops_p = sum(v[1] for v in verify_b)
    ver_tflops = ver_flops_p * args.steps / (ver_ms / 1e3) / 1e12
    stage_bytes_p = sum(sg.stage_bytes(gi) for gi in (0, 1))
    dom = max(kind_ms, key=kind_ms.get)
    dom_ms = kind_ms[dom] / kind_launch[dom]
    dom_alg = kind_bytes[dom] / kind_launch[dom]
    achieved = dom_alg / (dom_ms / 1e3) / 1e9
    kname = "draft_attn_kernel<128,%s,1>" % ("0" if dom == DROP else str(w.bits))
    total_kernel_ms = sum(kind_ms.values()) + ver_ms
    launches = sum(len(bt._steps) + bt.verify_launches() * args.head_chunks + 2 for bts in groups for bt in bts)
    overlap = statistics.mean(_covered(iv, comp_iv) for iv in copy_iv) if copy_iv else None
    if args.timeline:
        tl = [{"period": k, "host_issue_start_ms": host_t[k],
               "draft": [[rel(a), rel(b_)] for gi in (0, 1) for a, b_ in evs[k]["draft%d" % gi]],
               "verify": [[rel(evs[k]["verify%d" % gi][0]), rel(evs[k]["verify%d" % gi][1])] for gi in (0, 1)],
               "stage": [[rel(evs[k]["stage%d" % gi][0]), rel(evs[k]["stage%d" % gi][1])] for gi in (0, 1)]}
              for k in range(args.steps)]
        json.dump({"t_ms": t_ms, "steps": args.steps, "periods": tl}, open(args.timeline, "w"))

    # --- end to end through the engine's host-input period: every period copies each batch's
    # queries and drafted K/V rows, drafts, logits and L from pinned host memory and returns the
    # accepted tokens and counts to pinned host memory, besides staging the host-resident KV_full
    hrs = [[engine.HostRound(bt, *io[gi][j], names=("q", "k_new", "v_new")) for j, bt in enumerate(groups[gi])]
           for gi in (0, 1)]
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 50))
    for k in range(2):
        sg.period(None, host_rounds=hrs)
        if k == 0 and not args.no_graphs:
            sg.capture_drafts(host_rounds=hrs)
    torch.cuda.synchronize()
    f0, f1 = mk()
    torch.cuda.synchronize()
    f0.record(ks)
    cs.wait_event(f0)
    for _ in range(e2e_steps):
        sg.period(None, host_rounds=hrs)
    f1.record(ks)
    torch.cuda.synchronize()
    e2e_tokens = sum(int(hr.host_n_acc.sum().item()) for gi in (0, 1) for hr in hrs[gi])
    assert e2e_tokens == tokens, (e2e_tokens, tokens)
    h2d = stage_bytes_p + sum(hr.h2d_bytes for gi in (0, 1) for hr in hrs[gi])
    d2h = sum(hr.d2h_bytes for gi in (0, 1) for hr in hrs[gi])
    e2e = {"value": tokens * e2e_steps / (f0.elapsed_time(f1) / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "path": "engine.StaggeredOffload.period(host_rounds=...): round inputs from pinned host memory, "
                   "host-resident KV_full staged, accepted tokens and counts back to pinned host memory"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "Hq": w.Hq, "Hkv": w.Hkv, "d": d,
                       "ctx_min": min(w.ctx), "ctx_max": max(w.ctx), "ctx_mean": sum(w.ctx) / B,
                       "L_min": min(w.L), "L_max": w.L_max, "V": w.V, "bits": w.bits,
                       "requests_token_drop": sum(m == DROP for m in w.mode), "requests_on_host": sum(w.on_host),
                       "tokens_per_step": tokens, "groups": split, "head_chunks": args.head_chunks,
                       "host_issue_ms_per_step": host_ms / args.steps, "draft_graphs": not args.no_graphs,
                       "step": "one staggering period: every request drafts its L steps (one draft call per mode "
                               "and step), host-resident KV_full is staged, every request is verified and accepted",
                       "l2": "inputs larger than L2 (full KV %.1f GB, per draft step up to %.2f GB of KV_comp, logits "
                             "%.2f GB)" % (sum(full_b) / 1e9, max(kind_bytes[m] / kind_launch[m] for m in modes) / 1e9 * 1,
                                            logits.numel() * 4 / 1e9)},
            "e2e": e2e, "gpu_launches": launches * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": profiled_traffic(kname, w.name),
                         "kernel": kname + " (the largest GPU-time share of the period: one vc_draft_attn call; "
                                           "mean over every draft call of its mode in the timed periods)",
                         "algorithmic_bytes_per_launch": dom_alg, "avg_launch_ms": dom_ms, "peak_kind": peak_kind,
                         "share_of_kernel_time": kind_ms[dom] / total_kernel_ms},
            "kernels": {**{"draft_" + m: {"ms_per_step": kind_ms[m] / args.steps, "launches_per_step":
                                          kind_launch[m] // args.steps,
                                          "gbs": kind_bytes[m] / (kind_ms[m] / 1e3) / 1e9,
                                          "frac_of_hbm": kind_bytes[m] / (kind_ms[m] / 1e3) / 1e9 / hbm}
                           for m in modes},
                        "verify": {"ms_per_step": ver_ms / args.steps, "gbs": ver_bytes_p * args.steps / (ver_ms / 1e3) / 1e9,
                                   "frac_of_hbm": ver_bytes_p * args.steps / (ver_ms / 1e3) / 1e9 / hbm,
                                   "tflops": ver_tflops, "tensor_frac_of_bf16_sustained": ver_tflops / bf16,
                                   "flops_per_step": ver_flops_p,
                                   "note": "in-period intervals include waiting for the group's copy; 'alone' is "
                                           "the same work with nothing else running",
                                   "alone": {**ver_alone, "frac_of_hbm": ver_alone["gbs"] / hbm,
                                             "tensor_frac_of_bf16": ver_alone["tflops"] / float(peaks["bf16_tflops"])}}},
            "stage": {"bytes_per_step": stage_bytes_p, "gbs": stage_bytes_p * args.steps / (stage_ms / 1e3) / 1e9
                      if stage_ms else None, "link_alone_gbs": link_alone,
                      "frac_of_link": (stage_bytes_p * args.steps / (stage_ms / 1e3) / 1e9) / link_alone
                      if stage_ms and link_alone else None,
                      "copy_time_under_compute": overlap, "copy_ms_per_step": stage_ms / args.steps},
            "plan": {"modelled_period_ms": t_plan / 1e6, "rates_gbs": {**{"draft_" + m: rate[m] for m in modes},
                                                                     "verify": rate_v, "link": rate_s}},
            "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_oracle(w)
    print(json.dumps(line))
    return 0


def run_e2e(w, bt, draft, logits, L, out_tokens, n_acc, stream, steps, barrier, dist, world, device, quant=0):
    """Each step is one call of the engine's host-input round: that round's inputs (queries,
    drafted K/V, importance, drafts, logits, L) are copied from pinned host memory, the round runs
    through the C ABI, and n_acc and the accepted tokens are read back into pinned host memory.
    The accept inputs cross the host link on a second stream while the GPU drafts."""
    import torch
    from lossless_compressed_kv_vc_gb300 import engine
    hr = engine.HostRound(bt, logits, draft, L, out_tokens, n_acc,
                          names=("q", "k_new", "v_new") if quant else ("q", "k_new", "v_new", "importance"))
    copy_stream = torch.cuda.Stream()
    h2d, d2h = hr.h2d_bytes, hr.d2h_bytes

    def step():
        bt.run_round_from_host(hr, stream, copy_stream, compress=quant == 0)

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
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "offload":
        return run_offload(args)
    if args.workload == "stagger":
        return run_stagger(args)
    if args.workload == "importance":
        return run_importance(args)
    if args.workload == "mixed":
        return run_mixed(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main() or 0)
