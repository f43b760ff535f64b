#!/usr/bin/env python3
"""Benchmark of the batched speculative-decoding verify-and-sample step.

One step = one spec_verify_sample call over the whole serving-shaped batch
(B=64 sequences, gamma=5 drafts, V=128256 bf16 logits, temperature 0.7,
top-k 50, top-p 0.9 for target and draft), inputs resident in HBM.  The step
rotates over 4 independent input sets (4 x 180.6 MB, larger than the 126 MB
L2), so every call streams its logits from HBM.

Prints ONE JSON line (rank 0).  Metric: verified positions/s (target
positions consumed, sum of gamma_b + 1), next to the logits HBM GB/s of the
verify kernel as a fraction of the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (weak scaling: one batch per GPU,
                                                       no data-path collective)

--impl reference times the float64 CPU oracle (the only reference that exists
for this method) on the same workload, one sequence per step.
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

METRIC = "verified positions/s and logits HBM GB/s (% of peak), B=64 g=5 V=128256 bf16"
WID = 3             # the serving workload: the default, and the one METRIC names
SAMPLING_WIDS = (2, 3, 5)
GREEDY_WID = 4
L2_BYTES = 126 * 2 ** 20
ROTATE = 4
KERNEL_SOURCES = ["speculative_decoding_verification_44_gb300/csrc/spec_verify.cu",
                  "speculative_decoding_verification_44_gb300/csrc/sv_row.cuh",
                  "speculative_decoding_verification_44_gb300/csrc/sv_common.cuh"]
PROFILE = os.path.join(ROOT, "profiles", "sample_list_kernel_serving_B64_g5_V128256.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--lenience", type=float, default=None,
                    help="sampling workloads: spec_verify_sample_lenient with this beta")
    ap.add_argument("--eos", type=int, default=None,
                    help="sampling workloads: spec_verify_sample_ex with this end-of-sequence token")
    ap.add_argument("--per-seq-rules", action="store_true",
                    help="sampling workloads: spec_verify_sample_ex with the workload's rules given per sequence")
    ap.add_argument("--tree", action="store_true",
                    help="spec_verify_greedy_tree (greedy workload) or spec_verify_sample_tree (sampling "
                         "workloads) over draft trees of the same rows")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the steps as eager launches instead of one CUDA-graph replay")
    ap.add_argument("--workload", default="serving-zipf-topk-topp",
                    help="workload to time (default: the serving workload); the others exist for "
                         "profiling the full-row, small-vocabulary and greedy paths")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller cases for profiling; not a bench line)")
    ap.add_argument("--early-exit", action="store_true",
                    help="greedy: spec_verify_greedy_early; sampling: spec_verify_sample_ex with early_exit "
                         "(positions in order, rows after each sequence's stop skipped)")
    return ap.parse_args()


def workload_id(name: str) -> int:
    from speculative_decoding_verification_44_gb300 import workloads
    for wid in SAMPLING_WIDS + (GREEDY_WID,):
        if workloads.NAMES[wid] == name:
            return wid
    raise SystemExit(f"--workload must be one of {[workloads.NAMES[w] for w in SAMPLING_WIDS + (GREEDY_WID,)]}")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """dram bytes per launch from the committed ncu summary, if it matches the current kernel."""
    try:
        fields = {}
        with open(PROFILE) as f:
            for ln in f:
                if ":" in ln:
                    k, v = ln.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha") != kernel_source_sha():
            return None
        return float(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_draft_probs(rows, params):
    """Draft distribution q for drawing the benchmark's draft tokens (the library's transform)."""
    import speculative_decoding_verification_44_gb300 as sv
    probs, _ = sv.transform_probs(rows.contiguous(), params)
    return probs


def cpu_oracle_probs(rows, params):
    import numpy as np
    import oracle
    import torch
    p, _ = oracle.transform_rows(rows.float().double().numpy(), float(np.float32(params.temperature)),
                                 int(params.top_k), float(np.float32(params.top_p)))
    return torch.from_numpy(p)


def oracle_sample_time(w, seqs, budget_s=None):
    """Time the float64 oracle on the given sequences; returns (positions, seconds, n_seq)."""
    import numpy as np
    import oracle

    def f64(t):
        return t.detach().to("cpu").float().double().numpy()

    tp = (float(np.float32(w.target_params.temperature)), int(w.target_params.top_k),
          float(np.float32(w.target_params.top_p)))
    dp = (float(np.float32(w.draft_params.temperature)), int(w.draft_params.top_k),
          float(np.float32(w.draft_params.top_p)))
    gam = w.gamma_per_seq.cpu().numpy() if w.gamma_per_seq is not None else None
    oh = w.draft_is_onehot.cpu().numpy() if w.draft_is_onehot is not None else None
    positions, elapsed, n = 0, 0.0, 0
    seqs = list(seqs)
    if budget_s is not None:                  # cycle over the sequences until the budget is spent
        seqs = seqs * 1000
    for b in seqs:
        tl = f64(w.target_logits[b:b + 1])
        dl = f64(w.draft_logits[b:b + 1])
        toks = w.draft_tokens[b:b + 1].cpu().numpy()
        ua = w.u_accept[b:b + 1].cpu().double().numpy()
        us = w.u_sample[b:b + 1].cpu().double().numpy()
        g = gam[b:b + 1] if gam is not None else None
        o = oh[b:b + 1] if oh is not None else None
        t0 = time.perf_counter()
        oracle.verify_sample(tl, dl, toks, ua, us, tp, dp, gamma_per_seq=g, one_hot=o)
        elapsed += time.perf_counter() - t0
        positions += (int(g[0]) if g is not None else w.G) + 1
        n += 1
        if budget_s is not None and elapsed >= budget_s:
            break
    return positions, elapsed, n


def _oracle_one(args):
    """One sequence through the oracle (a worker of the all-cores baseline)."""
    import oracle
    tl, dl, toks, ua, us, tp, dp, g, o = args
    oracle.verify_sample(tl, dl, toks, ua, us, tp, dp, gamma_per_seq=g, one_hot=o)
    return (int(g[0]) if g is not None else toks.shape[1]) + 1


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                k = ln.split(":", 1)[0].strip().lower()
                if k in ("model name", "cpu model"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def oracle_sample_time_pool(w, seqs, budget_s=12.0):
    """The oracle on all host cores: a spawn-started process pool, one sequence per task.
    Returns (positions, seconds, sequences, workers)."""
    import multiprocessing as mp
    import numpy as np

    def f64(t):
        return t.detach().to("cpu").float().double().numpy()

    tp = (float(np.float32(w.target_params.temperature)), int(w.target_params.top_k),
          float(np.float32(w.target_params.top_p)))
    dp = (float(np.float32(w.draft_params.temperature)), int(w.draft_params.top_k),
          float(np.float32(w.draft_params.top_p)))
    gam = w.gamma_per_seq.cpu().numpy() if w.gamma_per_seq is not None else None
    oh = w.draft_is_onehot.cpu().numpy() if w.draft_is_onehot is not None else None
    workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    tasks = [(f64(w.target_logits[b:b + 1]), f64(w.draft_logits[b:b + 1]), w.draft_tokens[b:b + 1].cpu().numpy(),
              w.u_accept[b:b + 1].cpu().double().numpy(), w.u_sample[b:b + 1].cpu().double().numpy(), tp, dp,
              gam[b:b + 1] if gam is not None else None, oh[b:b + 1] if oh is not None else None) for b in seqs]
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_one, tasks[:workers])            # warm the workers (imports)
        positions, n = 0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:   # cycle over the sequences until the budget is spent
            chunk = [tasks[(n + i) % len(tasks)] for i in range(workers)]
            positions += sum(pool.map(_oracle_one, chunk))
            n += len(chunk)
        elapsed = time.perf_counter() - t0
    return positions, elapsed, n, workers


def outcome_stats(outs, sets, G):
    """Per-position empirical acceptance and the emitted-count histogram of the given outputs:
    acceptance at position i = P(draft i accepted | drafts before i accepted), over the
    sequences with gamma_b > i."""
    import torch
    acc_n = [0] * G
    acc_d = [0] * G
    hist = [0] * (G + 2)
    for o, w in zip(outs, sets):
        nacc = o.num_accepted.cpu().long()
        gb = (w.gamma_per_seq.cpu().long() if w.gamma_per_seq is not None
              else torch.full_like(nacc, G))
        for i in range(G):
            reach = (nacc >= i) & (gb > i)
            acc_d[i] += int(reach.sum())
            acc_n[i] += int((reach & (nacc > i)).sum())
        for e in (nacc[nacc >= 0] + 1).tolist():
            hist[e] += 1
    return {"acceptance_per_position": [round(n / d, 4) if d else None for n, d in zip(acc_n, acc_d)],
            "emitted_count_histogram": {str(k): v for k, v in enumerate(hist) if k >= 1},
            "sequences": sum(int(o.num_accepted.numel()) for o in outs)}


def replica_ids(rank: int, rotate: int = ROTATE) -> list[int]:
    """Input sets of one rank: independent batches, disjoint across ranks (weak scaling)."""
    return [rank * rotate + r for r in range(rotate)]


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (timing: the slowest rank defines the step)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * world / (ms_per_step / 1e3)


def params_of(w) -> dict:
    p = w.target_params
    return {"temperature": round(float(p.temperature), 6), "top_k": int(p.top_k), "top_p": round(float(p.top_p), 6)}


def variant_of(args) -> str:
    """Metric suffix naming a non-default call (empty for the plain call)."""
    parts = []
    if args.lenience is not None:
        parts.append(f"lenience {args.lenience}")
    if args.eos is not None:
        parts.append(f"eos {args.eos}")
    if args.per_seq_rules:
        parts.append("per-sequence rules")
    if getattr(args, "early_exit", False):
        parts.append("early exit")
    return f" ({', '.join(parts)})" if parts else ""


def metric_of(wid: int, w) -> str:
    if wid == WID:
        return METRIC
    dt = "bf16" if w.dtype.itemsize == 2 else "f32"
    return f"verified positions/s and logits HBM GB/s (% of peak), {w.name} B={w.B} g<={w.G} V={w.V} {dt}"


def run_reference(args, rank):
    """Reference arm: the float64 oracle on the host cores, one sequence per step."""
    if rank != 0:
        return
    from speculative_decoding_verification_44_gb300 import workloads
    wid = workload_id(args.workload)
    if wid == GREEDY_WID:
        raise SystemExit("the reference arm times the sampling oracle; use a sampling workload")
    w = workloads.make(wid, "cpu", draft_probs=cpu_oracle_probs)
    order = [s % w.B for s in range(args.warmup + args.steps)]
    oracle_sample_time(w, order[: args.warmup])
    pos, secs, n = oracle_sample_time(w, order[args.warmup:])
    value = pos / secs
    line = {
        "impl": "reference", "metric": metric_of(wid, w), "value": value, "unit": "positions/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, n), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"early_logits_reads": True, "workload": workloads.NAMES[wid], "B": w.B, "gamma": w.G, "V": w.V,
                   "dtype": "bf16" if w.dtype.itemsize == 2 else "f32", **params_of(w),
                   "step": "one sequence (gamma_b + 1 verified positions) per step"},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} sequences of the {workloads.NAMES[wid]} workload, one per step"},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_greedy(args, rank, world, dev, sv, workloads):
    """Greedy workload (all rows, or early exit): device-timed steps over rotating inputs."""
    import torch
    sets = [workloads.make(GREEDY_WID, dev, replica=rep, **({"B": args.batch} if args.batch else {}))
            for rep in replica_ids(rank)]
    w0 = sets[0]
    B, G, V = w0.B, w0.G, w0.V
    rt, _ = w0.rows_used()
    ws = sv.new_workspace(sv.greedy_workspace_size(B, G), dev)
    outs = [sv.alloc_outputs(B, G, dev, accept_prob=False, residual_z=False) for _ in range(ROTATE)]
    rows = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(ROTATE)]
    trees = []
    if args.tree:
        # draft trees over the same G + 1 rows: node i's parent is random among the earlier
        # nodes, its token the parent row's argmax with probability 0.8 (the workload's rate)
        import numpy as np
        ws = sv.new_workspace(sv.tree_workspace_size(B, G + 1), dev)
        for r, w in enumerate(sets):
            rng = np.random.default_rng(5000 + r)
            arg = w.target_logits.float().argmax(dim=-1).cpu().numpy()
            tok = np.zeros((B, G + 1), dtype=np.int32)
            par = np.full((B, G + 1), -1, dtype=np.int32)
            for b in range(B):
                for i in range(1, G + 1):
                    par[b, i] = rng.integers(0, i)
                    tok[b, i] = arg[b, par[b, i]] if rng.random() < 0.8 else rng.integers(0, V)
            trees.append((torch.from_numpy(tok).to(dev), torch.from_numpy(par).to(dev),
                          torch.empty(B, G + 1, dtype=torch.int32, device=dev)))
            outs[r] = sv.VerifyOutput(tokens=torch.empty(B, G + 1, dtype=torch.int32, device=dev),
                                      num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                                      status=torch.empty(B, dtype=torch.int32, device=dev))

    def step(i):
        w, r = sets[i % ROTATE], i % ROTATE
        if args.tree:
            tok, par, path = trees[r]
            sv.verify_greedy_tree(w.target_logits, tok, par, workspace=ws, out=outs[r], path=path)
        elif args.early_exit:
            sv.verify_greedy_early(w.target_logits, w.draft_tokens, w.gamma_per_seq, workspace=ws, out=outs[r],
                                   rows_read=rows[r])
        else:
            sv.verify_greedy(w.target_logits, w.draft_tokens, w.gamma_per_seq, workspace=ws, out=outs[r])

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    K = args.steps
    stream = torch.cuda.current_stream()
    with ClockSampler(torch.cuda.current_device()) as clk:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    ms_per_step = max_over_ranks(t0.elapsed_time(t1), world, dev) / K
    row_bytes = V * w0.target_logits.element_size()
    read = [int(r.sum().item()) for r in rows] if (args.early_exit and not args.tree) else [rt] * ROTATE
    needed = [int((o.num_accepted.clamp(min=0) + 1).sum().item()) for o in outs]
    peak, peak_kind = measured_peaks()
    # algorithmic rows: every row for the all-rows verifier (it checks them all), the rows
    # up to each sequence's stop for early exit (speculative extra reads are waste)
    alg_rows = statistics.mean(needed) if (args.early_exit and not args.tree) else rt
    achieved = alg_rows * row_bytes / (ms_per_step / 1e3) / 1e9
    if rank == 0:
        line = {
            "metric": f"verified positions/s, {w0.name} B={B} g={G} V={V} bf16"
                      + (" (draft trees of the same rows)" if args.tree else
                         " (early exit)" if args.early_exit else ""),
            "value": whole_job_rate(rt, world, ms_per_step), "unit": "positions/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"early_logits_reads": True, "workload": w0.name, "B": B, "gamma": G, "V": V, "early_exit": bool(args.early_exit), "tree": bool(args.tree),
                       "l2": f"inputs rotate over {ROTATE} independent sets of {rt * row_bytes / 1e6:.1f} MB"},
            "rows_read_per_step": statistics.mean(read), "rows_needed_per_step": statistics.mean(needed),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_kind": f"of {peak_kind}",
                         "kernel": "sv::greedy_tree_kernel<bf16>" if args.tree else
                                   "sv::greedy_early_kernel<bf16>" if args.early_exit else "sv::greedy_kernel<bf16>",
                         "algorithmic_bytes_per_launch": alg_rows * row_bytes,
                         "bytes_read_per_launch": statistics.mean(read) * row_bytes},
            "cpu_baseline": None, "e2e": None, "gpu_launches": K, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def run_sample_tree(args, rank, world, dev, sv, workloads, wid):
    """Sampling workloads as draft trees over the same rows (spec_verify_sample_tree): node c of
    sequence b (c = 1..G) gets a random earlier parent and a token drawn from the draft distribution
    at that parent; node c's target row is the workload's target row c, its draft row draft row c
    (the last node's draft row is never read: it has no children)."""
    import torch
    sets = [workloads.make(wid, dev, draft_probs=gpu_draft_probs, replica=rep,
                           **({"B": args.batch} if args.batch else {})) for rep in replica_ids(rank)]
    w0 = sets[0]
    B, G, V = w0.B, w0.G, w0.V
    N = G + 1
    esize = w0.target_logits.element_size()
    trees = []
    alg = []
    for r, w in enumerate(sets):
        gen = torch.Generator(device=dev).manual_seed(6000 + 100 * rank + r)
        q, _ = sv.transform_probs(w.draft_logits.reshape(B * G, V).contiguous(), w.draft_params)
        q = q.view(B, G, V)
        par = torch.full((B, N), -1, dtype=torch.int32, device=dev)
        tok = torch.zeros(B, N, dtype=torch.int32, device=dev)
        for c in range(1, N):
            pc = torch.floor(torch.rand(B, generator=gen, device=dev) * c).long().clamp(max=c - 1)
            par[:, c] = pc.int()
            tok[:, c] = torch.multinomial(q[torch.arange(B, device=dev), pc], 1, generator=gen).squeeze(1).int()
        dft = torch.cat([w.draft_logits, torch.zeros_like(w.draft_logits[:, :1])], dim=1).contiguous()
        u_node = torch.cat([torch.zeros(B, 1, device=dev), w.u_accept], dim=1).contiguous()
        has_child = torch.zeros(B, N, dtype=torch.bool, device=dev)
        has_child.scatter_(1, par[:, 1:].long(), True)
        alg.append(int((N + has_child.sum(dim=1)).sum().item()) * V * esize)
        trees.append((w.target_logits, dft, tok, par, u_node, w.u_sample))
    ws = sv.new_workspace(sv.tree_sample_workspace_size(B, N, V, w0.target_params, w0.draft_params), dev)
    outs = []
    for _ in range(ROTATE):
        outs.append(sv.VerifyOutput(tokens=torch.empty(B, N, dtype=torch.int32, device=dev),
                                    num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                                    status=torch.empty(B, dtype=torch.int32, device=dev),
                                    accept_prob=torch.empty(B, N - 1, dtype=torch.float32, device=dev),
                                    residual_z=torch.empty(B, dtype=torch.float32, device=dev)))
    paths = [torch.empty(B, N, dtype=torch.int32, device=dev) for _ in range(ROTATE)]

    def step(i, stream=None):
        r = i % ROTATE
        t = trees[r]
        sv.verify_sample_tree(*t, w0.target_params, w0.draft_params, workspace=ws, out=outs[r], path=paths[r],
                              stream=stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    K = args.steps
    stream = torch.cuda.current_stream()
    graph = g_ev = None
    if not args.no_graph:
        # K calls captured as one CUDA graph, timed by event-record nodes inside it
        gstream = torch.cuda.Stream()
        gstream.wait_stream(stream)
        with torch.cuda.stream(gstream):
            for i in range(ROTATE):
                step(i, gstream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        try:
            g_ev = (torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True))
        except TypeError:
            g_ev = None
        with torch.cuda.graph(graph, stream=gstream):
            if g_ev is not None:
                g_ev[0].record(gstream)
            for i in range(K):
                step(i, gstream)
            if g_ev is not None:
                g_ev[1].record(gstream)
        graph.replay()
        torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    total_ms = g_ev[0].elapsed_time(g_ev[1]) if g_ev is not None else t0.elapsed_time(t1)
    ms_per_step = max_over_ranks(total_ms, world, dev) / K
    peak, peak_kind = measured_peaks()
    alg_bytes = statistics.mean(alg)
    achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
    depth = statistics.mean(float(o.num_accepted.float().mean().item()) for o in outs)
    if rank == 0:
        dname = "bf16" if esize == 2 else "f32"
        line = {
            "metric": metric_of(wid, w0) + " (draft trees of the same rows)",
            "value": whole_job_rate(B * N, world, ms_per_step), "unit": "tree nodes/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dname, "data": "synthetic",
            "config": {"early_logits_reads": True, "workload": w0.name, "B": B, "nodes": N, "V": V, **params_of(w0), "tree": True,
                       "l2": f"inputs rotate over {ROTATE} independent sets",
                       "launch": ("K eager launches" if graph is None else
                                  "K steps as one CUDA graph replay" + (", timed by event-record nodes inside the graph"
                                                                        if g_ev is not None else ""))},
            "accepted_path_length_mean": depth,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "peak_kind": f"of {peak_kind}", "kernel": f"sv::sample_tree_kernel<{dname}>",
                         "algorithmic_bytes_per_launch": alg_bytes},
            "cpu_baseline": None, "e2e": None, "gpu_launches": K, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from speculative_decoding_verification_44_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads

    # every call here reads logits that were written before the timed region (or
    # copied in by the e2e leg), so the verifiers may stream them before waiting
    # for the previous call: back-to-back calls overlap
    sv.set_early_logits_reads(True)

    # independent batches: replica = rank * ROTATE + r
    wid = workload_id(args.workload)
    if wid == GREEDY_WID:
        run_greedy(args, rank, world, dev, sv, workloads)
        return
    if args.tree:
        run_sample_tree(args, rank, world, dev, sv, workloads, wid)
        return
    sets = [workloads.make(wid, dev, draft_probs=gpu_draft_probs, replica=rep,
                           **({"B": args.batch} if args.batch else {})) for rep in replica_ids(rank)]
    w0 = sets[0]
    B, G, V = w0.B, w0.G, w0.V
    rt, rd = w0.rows_used()
    esize = w0.target_logits.element_size()
    logits_bytes = (rt + rd) * V * esize
    # a target row without a small top-k takes the full-row path; its draw is a second kernel
    full_target = not (1 <= w0.target_params.top_k <= 128 and w0.target_params.top_k < V)
    io_bytes = B * G * 4 * 2 + B * 4 + B * (G + 1) * 4 + B * 4 * 3 + B * G * 4
    alg_bytes = logits_bytes + io_bytes
    # optional paths: lenience, end-of-sequence commit, per-sequence rules (the workload's own
    # rule for every sequence; promised kept-list when that rule is on the kept-list path)
    kept = not full_target and 1 <= w0.draft_params.top_k <= 128
    opts = dict(lenience=args.lenience, eos_token=args.eos)
    if args.early_exit:
        opts["early_exit"] = True
    if args.per_seq_rules:
        opts.update(target_rules=[w0.target_params] * B, draft_rules=[w0.draft_params] * B, kept_list_only=kept)
        if not kept:
            full_target = True
    ws = sv.new_workspace(sv.workspace_size(B, G, V, w0.target_params, w0.draft_params,
                                            per_sequence=args.per_seq_rules, kept_list_only=kept), dev)
    outs = [sv.alloc_outputs(B, G, dev) for _ in range(ROTATE)]
    stream = torch.cuda.current_stream()

    calls = [sv.BoundSample(w.target_logits, w.draft_logits, w.draft_tokens, w.u_accept, w.u_sample,
                            w.target_params, w.draft_params, gamma_per_seq=w.gamma_per_seq,
                            draft_is_onehot=w.draft_is_onehot, workspace=ws, out=outs[r], **opts)
             for r, w in enumerate(sets)]

    def step(i):
        calls[i % ROTATE]()

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    graph = None
    g_ev = None
    if not args.no_graph:
        # the same K calls captured once as a CUDA graph (serving loops replay graphs:
        # no host launch gap between steps); each call is still one C-ABI launch
        gstream = torch.cuda.Stream()
        gcalls = [sv.BoundSample(w.target_logits, w.draft_logits, w.draft_tokens, w.u_accept, w.u_sample,
                                 w.target_params, w.draft_params, gamma_per_seq=w.gamma_per_seq,
                                 draft_is_onehot=w.draft_is_onehot, workspace=ws, out=outs[r], stream=gstream,
                                 **opts)
                  for r, w in enumerate(sets)]
        gstream.wait_stream(stream)
        with torch.cuda.stream(gstream):
            for i in range(ROTATE):
                gcalls[i]()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        # timing events recorded inside the graph (event-record nodes): the region is
        # the K steps' device work, without the host's graph launch latency
        try:
            g_ev = (torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True))
        except TypeError:
            g_ev = None
        with torch.cuda.graph(graph, stream=gstream):
            if g_ev is not None:
                g_ev[0].record(gstream)
            for i in range(K):
                gcalls[i % ROTATE]()
            if g_ev is not None:
                g_ev[1].record(gstream)
        graph.replay()
        torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        # per-launch kernel durations (eager launches, events around each) for the roofline
        torch.cuda.synchronize()
        for i in range(K):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        # the timed region: K steps, one graph replay (or K eager launches)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                step(i)
        t_all1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        in_graph_ms = g_ev[0].elapsed_time(g_ev[1]) if g_ev is not None else None
        # spread: the same K-step region repeated until >= 200 calls and >= 0.5 s, each
        # repetition timed on the device (per-step times: median, p10, p90)
        rep_ms = []
        r_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        t_spread = time.perf_counter()
        while len(rep_ms) < 4096 and (len(rep_ms) * K < 200 or time.perf_counter() - t_spread < 0.5):
            r_ev[0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                for i in range(K):
                    step(i)
            r_ev[1].record(stream)
            torch.cuda.synchronize()
            ev_pair = g_ev if g_ev is not None else r_ev
            rep_ms.append(ev_pair[0].elapsed_time(ev_pair[1]) / K)
    rep_ms.sort()
    # one call alone: a graph of a single call per rotation set (events inside it),
    # replayed with a synchronize between replays -- the latency of one verify with no
    # neighbouring call to overlap (back-to-back calls overlap: a call streams its rows
    # before it waits for the previous call in the stream)
    single_ms = None
    if graph is not None and g_ev is not None:
        g1 = []
        for r in range(ROTATE):
            ev1 = (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True))
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=gstream):
                ev1[0].record(gstream)
                gcalls[r]()
                ev1[1].record(gstream)
            g1.append((gr, ev1))
        torch.cuda.synchronize()
        single = []
        for t in range(4 * ROTATE + 32):
            gr, ev1 = g1[t % ROTATE]
            gr.replay()
            torch.cuda.synchronize()
            if t >= 2 * ROTATE:
                single.append(ev1[0].elapsed_time(ev1[1]))
        single_ms = max_over_ranks(statistics.median(single), world, dev)

    def pct(v, q):
        return v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]

    spread = {"repetitions": len(rep_ms), "calls": len(rep_ms) * K, "ms_per_step_median": pct(rep_ms, 0.5),
              "ms_per_step_p10": pct(rep_ms, 0.1), "ms_per_step_p90": pct(rep_ms, 0.9)}
    outer_ms = t_all0.elapsed_time(t_all1)
    total_ms = in_graph_ms if in_graph_ms is not None else outer_ms
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / K
    value = whole_job_rate(rt, world, ms_per_step)

    # outcome statistics of the last step (emitted tokens / s etc.)
    last = outs[(K - 1) % ROTATE]
    emitted = int((last.num_accepted.clamp(min=-1) + 1).sum().item())

    peak, peak_kind = measured_peaks()
    # average launch duration over the timed region: the graph replay's K back-to-back
    # launches (events around one eager launch also hold its launch latency)
    avg_launch_s = (total_ms / K if graph is not None else statistics.mean(launch_ms)) / 1e3
    if args.early_exit:
        # early exit: the bytes a sequential verifier needs -- target rows 0..j and draft
        # rows 0..min(j, gamma_b - 1) of each sequence -- averaged over the rotation sets
        needed = []
        for r, w in enumerate(sets):
            j = outs[r].num_accepted.long().clamp(min=0)
            gb = w.gamma_per_seq.long() if w.gamma_per_seq is not None else torch.full_like(j, G)
            model = (torch.ones_like(j, dtype=torch.bool) if w.draft_is_onehot is None
                     else w.draft_is_onehot == 0) if w.draft_logits is not None else torch.zeros_like(j, dtype=torch.bool)
            rows = (j + 1) + torch.where(model, torch.minimum(j + 1, gb), torch.zeros_like(j))
            needed.append(int(rows.sum().item()) * V * esize + io_bytes)
        alg_bytes = statistics.mean(needed)
    achieved = alg_bytes / avg_launch_s / 1e9
    traffic = profile_traffic() if wid == WID else None
    dname = "bf16" if esize == 2 else "f32"
    # the kept-list kernel serves the plain and lenient calls when every row is on the
    # streaming top-k path, rows are 16-byte aligned and each sequence's row blocks
    # fit its gather buffer (the library's own dispatch rule)
    tk, dk = int(w0.target_params.top_k), int(w0.draft_params.top_k)
    kcap = max(tk, dk if w0.draft_logits is not None else 0)
    list_path = (not args.early_exit and args.eos is None and not args.per_seq_rules and not full_target
                 and (w0.draft_logits is None or 1 <= dk <= 128 and dk < V) and (V * esize) % 16 == 0
                 and G <= 31 and (2 * G + 1) * (1 + kcap) <= 1024)
    kname = (f"sv::sample_list_kernel<{dname}>" if list_path else f"sv::sample_kernel<{dname}>"
             + (f" + sv::draw_kernel<{dname}>" if full_target else ""))
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "peak_kind": f"of {peak_kind}",
                "kernel": kname, "algorithmic_bytes_per_launch": alg_bytes,
                "launch_ms_avg_timed_region": avg_launch_s * 1e3,
                "launch_ms_median_eager": statistics.median(launch_ms),
                "frac_of_nominal_8TBps": achieved / 8000.0}
    if single_ms is not None:
        roofline["single_call"] = {"ms_median": single_ms,
                                   "frac": alg_bytes / (single_ms / 1e3) / 1e9 / peak,
                                   "how": "one call alone: a one-call graph per rotation set, events inside it, "
                                          "a synchronize between replays"}

    # end to end through the public API with host buffers (pinned), rank-local
    e2e = None
    if not args.no_e2e:
        w = sets[0]
        names = ["target_logits", "draft_logits", "draft_tokens", "u_accept", "u_sample"]
        names += [k for k in ("gamma_per_seq", "draft_is_onehot") if getattr(w, k) is not None]
        host = {k: getattr(w, k).cpu().pin_memory() for k in names}
        dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
        hout = {"tokens": torch.empty(B, G + 1, dtype=torch.int32).pin_memory(),
                "num_accepted": torch.empty(B, dtype=torch.int32).pin_memory(),
                "status": torch.empty(B, dtype=torch.int32).pin_memory()}
        dout = sv.alloc_outputs(B, G, dev, accept_prob=False, residual_z=False)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(v.numel() * v.element_size() for v in hout.values())

        def e2e_step():
            for k in host:
                dbuf[k].copy_(host[k], non_blocking=True)
            sv.verify_sample(dbuf["target_logits"], dbuf["draft_logits"], dbuf["draft_tokens"],
                             dbuf["u_accept"], dbuf["u_sample"], w.target_params, w.draft_params,
                             gamma_per_seq=dbuf.get("gamma_per_seq"), draft_is_onehot=dbuf.get("draft_is_onehot"),
                             workspace=ws, out=dout, **({"early_exit": True} if args.early_exit else {}))
            hout["tokens"].copy_(dout.tokens, non_blocking=True)
            hout["num_accepted"].copy_(dout.num_accepted, non_blocking=True)
            hout["status"].copy_(dout.status, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        Ke = max(5, min(K, 30))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / Ke
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": whole_job_rate(rt, world, e_ms), "unit": "positions/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pos, secs, n = oracle_sample_time(w0, list(range(B)), budget_s=10.0)
        single = {"value": pos / secs, "unit": "positions/s", "cores": 1,
                  "sample": f"{n} sequence verifications cycling over the {B} sequences of the same workload "
                            f"(rotation set 0), {pos} verified positions in {secs:.1f} s"}
        ppos, psecs, pn, workers = oracle_sample_time_pool(w0, list(range(B)), budget_s=10.0)
        cpu_baseline = {"value": ppos / psecs, "unit": "positions/s", "cores": workers, "kind": "oracle",
                        "sample": f"{pn} sequence verifications cycling over the {B} sequences of the same "
                                  f"workload (rotation set 0), one per task on a {workers}-process pool, "
                                  f"{ppos} verified positions in {psecs:.1f} s",
                        "cpu": cpu_model(), "single_core": single}

    if rank == 0:
        line = {
            "metric": metric_of(wid, w0) + variant_of(args), "value": value, "unit": "positions/s",
            "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dname, "data": "synthetic",
            "config": {"early_logits_reads": True, "workload": workloads.NAMES[wid], "B": B, "gamma": G, "V": V,
                       **params_of(w0), "batches_per_gpu": 1, "early_exit": bool(args.early_exit),
                       "l2": f"inputs rotate over {ROTATE} independent sets of {logits_bytes / 1e6:.1f} MB "
                             f"(each larger than the {L2_BYTES / 2**20:.0f} MiB L2)",
                       "parallelism": f"replicas x{world} (one batch per GPU, no data-path collective)",
                       "launch": ("K steps as one CUDA graph replay, timed by event-record nodes inside the graph"
                                  if g_ev is not None else
                                  "K steps as one CUDA graph replay" if graph is not None else "K eager launches")
                                 + "; early logits reads on (spec_set_early_logits_reads): a kept-list call "
                                   "streams its rows before it waits for the previous call, so consecutive calls "
                                   "overlap; roofline from the timed region's average time per call, single_call "
                                   "from one call alone"},
            "ms_per_step_with_graph_launch": outer_ms / K,
            "spread": spread,
            "sequences_per_s": B * world / (ms_per_step / 1e3),
            "drafts_judged_per_s": B * G * world / (ms_per_step / 1e3),
            "emitted_tokens_per_s_last_step": emitted * world / (ms_per_step / 1e3),
            "outcomes": outcome_stats(outs, sets, G),
            "logits_bytes_per_verified_position": logits_bytes / rt,
            "dram_bytes_per_verified_position": (traffic / rt) if traffic else None,
            "roofline": roofline, "cpu_baseline": cpu_baseline, "e2e": e2e,
            "gpu_launches": K * (2 if full_target else 1),
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
