"""Throughput of the speculative-sampling verify step on GB300.

One step = one verify call over one synthetic batch: B = 256 sequences with a
ragged lookahead gamma ~ U{1..10}, V = 152064, bf16 logits, T = 0.7, sampling
mode (one fused launch: plan, row statistics of the rows the result needs
-- rows after a sequence's first rejection are not read --, accept tests,
residual/bonus draw). The HBM figures count the per-call logit bytes of the
step, every row once (sum_b (2 gamma_b + 1) V elem); the ``roofline`` record
also gives the fraction on the bytes the result needs and the ncu traffic.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0). ``value`` is verified draft tokens per second
over all ranks (each rank verifies its own batch: weak scaling, no data-path
collective). Inputs are larger than L2 (two alternating batches of 0.93 GB
each), so no flush is needed between steps. ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/s (B×gamma per call) and achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
BENCH_CFG = 3
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batches", type=int, default=2, choices=[1, 2],
                    help="alternating input batches (2 keeps consecutive steps off L2)")
    ap.add_argument("--mode", default="sampling",
                    choices=["sampling", "greedy", "lossy", "restricted", "stats", "features"],
                    help="sampling verify (default), the greedy exact-match verify, the lossy "
                         "verify (f_sq lenience, eps 0.5), the restricted verify (top-k 20, "
                         "top-p 0.95 per sequence), or the row diagnostics: per-position "
                         "acceptance statistics (beta, TVD) or draft features (entropy, top-10)")
    ap.add_argument("--config", type=int, default=BENCH_CFG, choices=[0, 1, 2, 3, 4],
                    help="workload (default: the ragged B=256 bf16 batch; the others serve "
                         "profiling and the per-workload table)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, secs):
    """Whole-job verified tokens/s: every rank verifies its own batch of
    tokens_per_rank draft tokens (weak scaling) within the slowest rank's
    time secs."""
    return world * tokens_per_rank / secs


def workload_config(cfg, batch, mode):
    lb = batch.logit_bytes(greedy=mode == "greedy")
    g = cfg["gamma"]
    gdesc = (f"uniform {g[0]}..{g[1]} per sequence" if isinstance(g, (tuple, list)) else g)
    return {"workload": cfg["name"], "B": cfg["B"], "gamma": gdesc,
            "V": cfg["V"], "logit_dtype": cfg["dtype"], "temperature": cfg["T"], "mode": mode,
            "logit_bytes_per_step": batch.logit_bytes(greedy=mode == "greedy"),
            "draft_tokens_per_step": batch.draft_token_count(),
            "l2": ("inputs larger than L2: two alternating batches of %.2f GB"
                   % (lb / 1e9)) if lb > 129e6 else
                  ("inputs fit in L2 (%.1f MB a batch): a latency figure, not a bandwidth one"
                   % (lb / 1e6))}


def kernel_hash():
    """Hash of every kernel source: a stored traffic figure is used only while it matches."""
    hsh = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_token_gb300", "csrc")
    # the sources the fused sampling kernel is built from
    for name in ("sv_common.cuh", "sv_draw.cuh", "sv_fused.cu", "sv_internal.h", "sv_stream.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()[:16]


def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on a bounded sample of the same workload."""
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from speculative_decoding_token_gb300 import workload
    cfg = workload.CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    batch = workload.make_batch(args.config, device=dev)
    sample = list(range(16))
    a = workload.to_host_arrays(batch, sample)
    tokens = int(a["gamma"].sum())
    T = float(np.float32(batch.T))
    cores = max(1, min(os.cpu_count() or 1, 64))
    for w in range(args.warmup):
        oracle.verify_batch(a["target"], a["draft"], a["p_row_off"], a["q_row_off"],
                            a["draft_tokens"], a["gamma"], T, seed=w, seq_ids=a["seq_ids"],
                            nthreads=cores)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.verify_batch(a["target"], a["draft"], a["p_row_off"], a["q_row_off"],
                            a["draft_tokens"], a["gamma"], T, seed=1000 + s,
                            seq_ids=a["seq_ids"], nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, batch, "sampling"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"sequences 0..{len(sample) - 1} of the batch "
                                       f"({tokens} draft tokens) per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(batch, cores, greedy=False):
    """Oracle wall time for one full step of the workload on the host cores."""
    import numpy as np

    import oracle
    from speculative_decoding_token_gb300 import workload
    a = workload.to_host_arrays(batch)
    T = float(np.float32(batch.T))
    t0 = time.perf_counter()
    if greedy:
        oracle.verify_batch(a["target"], None, a["p_row_off"], None, a["draft_tokens"],
                            a["gamma"], 0.0, nthreads=cores)
    else:
        oracle.verify_batch(a["target"], a["draft"], a["p_row_off"], a["q_row_off"],
                            a["draft_tokens"], a["gamma"], T, seed=1, nthreads=cores)
    dt = time.perf_counter() - t0
    tokens = int(a["gamma"].sum())
    # the same oracle on one core, on a bounded sample of the batch
    sample = list(range(min(len(a["gamma"]), 16)))
    s = workload.to_host_arrays(batch, sample)
    t1 = time.perf_counter()
    if greedy:
        oracle.verify_batch(s["target"], None, s["p_row_off"], None, s["draft_tokens"],
                            s["gamma"], 0.0, seq_ids=s["seq_ids"], nthreads=1)
    else:
        oracle.verify_batch(s["target"], s["draft"], s["p_row_off"], s["q_row_off"],
                            s["draft_tokens"], s["gamma"], T, seed=1, seq_ids=s["seq_ids"],
                            nthreads=1)
    dt1 = time.perf_counter() - t1
    tok1 = int(s["gamma"].sum())
    return {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one whole step: all {len(a['gamma'])} sequences ({tokens} draft "
                      f"tokens), {dt:.2f} s",
            "one_core": {"value": tok1 / dt1, "unit": UNIT, "cores": 1,
                         "ms_per_step": dt1 / max(tok1, 1) * tokens * 1e3,
                         "sample": f"sequences 0..{len(sample) - 1} ({tok1} draft tokens), "
                                   f"{dt1:.2f} s, scaled to the whole step"},
            "ms_per_step": dt * 1e3}


def run_diagnostics(args, rank, world, local):
    """Times the row diagnostics on the workload: acceptance statistics of every
    position (both rows read, the second pass mostly from L2) or the draft
    features of every draft row (one pass). HBM figures count each row once."""
    import torch

    import speculative_decoding_token_gb300 as sv
    from speculative_decoding_token_gb300 import workload

    sv.build()
    cfg = workload.CONFIGS[args.config]
    batches = [workload.make_batch(args.config, device="cuda", seed=cfg["seed"] + 100 * rank + k)
               for k in range(args.batches)]
    h = sv.SpecVerify(cfg["B"], batches[0].gamma_max, cfg["V"])
    stream = torch.cuda.current_stream()
    stats = args.mode == "stats"
    B, gm = cfg["B"], batches[0].gamma_max
    beta = torch.empty(B, max(gm, 1), device="cuda")
    tvd = torch.empty_like(beta)
    nq = max(b.draft.shape[0] for b in batches)
    ent = torch.empty(nq, device="cuda")
    prob = torch.empty(nq, 10, device="cuda")
    idx = torch.empty(nq, 10, dtype=torch.int32, device="cuda")
    structs = [sv.make_batch_struct(b.target, b.draft, b.p_row_off, b.q_row_off,
                                    b.draft_tokens, b.gamma) for b in batches]

    def step(i):
        b = batches[i % len(batches)]
        if stats:
            sv.specverify_acceptance_stats(h.h, structs[i % len(batches)], cfg["T"], beta, tvd,
                                           stream=stream)
        else:
            sv.specverify_row_features(h.h, b.draft, cfg["T"], 10, ent, prob, idx,
                                       stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.25)
        start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        stop.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.05)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world)
    status = h.device_status()
    h.close()
    timed = [batches[i % len(batches)] for i in range(args.warmup, args.warmup + args.steps)]
    esz = batches[0].target.element_size()
    units = sum(b.draft_token_count() for b in timed)  # positions, or draft rows
    bytes_ = sum((2 if stats else 1) * b.draft_token_count() * b.V * esz for b in timed)
    secs = ms / 1e3
    peak, peak_kind = peaks()
    if rank != 0:
        return
    gbs = bytes_ / secs / 1e9
    line = {"metric": "positions/s (acceptance statistics)" if stats else
            "draft rows/s (entropy and top-10)", "value": world * units / secs,
            "unit": "positions/s" if stats else "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {**workload_config(cfg, batches[0], "sampling"), "mode": args.mode},
            "roofline": {"bound": "hbm",
                         "kernel": "pair_kernel" if stats else "features_rows_kernel + features_final_kernel",
                         "achieved": gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": bytes_ / args.steps,
                         "algorithmic_bytes": "every p_i and q_i row of a position once"
                         if stats else "every draft row once"},
            "clocks": clocks.summary(), "gpu_launches": args.steps, "device_status": status}
    print(json.dumps(line), flush=True)


RESTRICT_TOPK, RESTRICT_TOPP = 20, 0.95


def restricted_drafts(batch, T, k, top_p, seed):
    """Input preparation (not timed): draft tokens drawn from the top-k / top-p
    restricted draft rows, as a drafter with the same sampling settings emits
    them."""
    import torch
    gen = torch.Generator(device=batch.draft.device)
    gen.manual_seed(seed)
    toks = torch.zeros_like(batch.draft_tokens)
    g = batch.gamma.to(torch.int64)
    if batch.draft.shape[0] == 0:
        return toks
    v, i = torch.topk(batch.draft.float(), k, dim=1)
    w = torch.softmax(v / T, dim=1)
    before = torch.cumsum(w, 1) - w
    w = torch.where(before < top_p, w, torch.zeros_like(w))
    x = i.gather(1, torch.multinomial(w, 1, generator=gen)).flatten().to(torch.int32)
    seq = torch.repeat_interleave(torch.arange(batch.B, device=g.device), g)
    pos = torch.arange(x.numel(), device=g.device) - batch.q_row_off[seq]
    toks[seq, pos] = x
    return toks


def run_restricted(args, rank, world, local):
    """Times the restricted verify (per-sequence temperature, top-k, top-p) on
    the workload: every row of every sequence is read once."""
    import torch

    import speculative_decoding_token_gb300 as sv
    from speculative_decoding_token_gb300 import workload

    sv.build()
    cfg = workload.CONFIGS[args.config]
    batches = [workload.make_batch(args.config, device="cuda", seed=cfg["seed"] + 100 * rank + k)
               for k in range(args.batches)]
    B = cfg["B"]
    h = sv.SpecVerify(B, max(batches[0].gamma_max, 1), cfg["V"])
    stream = torch.cuda.current_stream()
    T = torch.full((B,), cfg["T"], dtype=torch.float32, device="cuda")
    k = torch.full((B,), RESTRICT_TOPK, dtype=torch.int32, device="cuda")
    p = torch.full((B,), RESTRICT_TOPP, dtype=torch.float32, device="cuda")
    for j, b in enumerate(batches):
        b.draft_tokens = restricted_drafts(b, cfg["T"], RESTRICT_TOPK, RESTRICT_TOPP, 7 + j)
    structs = [sv.make_batch_struct(b.target, b.draft, b.p_row_off, b.q_row_off,
                                    b.draft_tokens, b.gamma) for b in batches]
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    toks = torch.empty(B, batches[0].gamma_max + 1, dtype=torch.int32, device="cuda")
    h.set_timing(True)

    def step(i):
        sv.specverify_verify_restricted(h.h, structs[i % len(batches)], T, k, p, 1000 + i, n,
                                        toks, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    h.get_timing(sv.KERNEL_RESTRICT_ROWS, reset=True)  # (a reset clears every kernel's totals)
    barrier(world)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.25)
        start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        stop.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.05)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world)
    plan_ms, plan_n = h.get_timing(sv.KERNEL_RESTRICT_PLAN)
    fin_ms, fin_n = h.get_timing(sv.KERNEL_RESTRICT_FINAL)
    main_ms, main_n = h.get_timing(sv.KERNEL_RESTRICT_ROWS, reset=True)
    status = h.device_status()
    h.close()
    timed = [batches[i % len(batches)] for i in range(args.warmup, args.warmup + args.steps)]
    units = sum(b.draft_token_count() for b in timed)
    bytes_ = sum(b.logit_bytes() for b in timed)
    secs = ms / 1e3
    peak, peak_kind = peaks()
    if rank != 0:
        return
    kernel_gbs = bytes_ / (main_ms / 1e3) / 1e9
    line = {"metric": METRIC, "value": world * units / secs, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {**workload_config(cfg, batches[0], "sampling"), "mode": "restricted",
                       "top_k": RESTRICT_TOPK, "top_p": RESTRICT_TOPP},
            "hbm_gbs_per_gpu": bytes_ / secs / 1e9,
            "roofline": {"bound": "hbm", "kernel": "restrict_rows_kernel", "achieved": kernel_gbs,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": kernel_gbs / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": bytes_ / args.steps,
                         "algorithmic_bytes": "sum_b (2 gamma_b + 1) V elem: every row once",
                         "kernel_us": main_ms / main_n * 1e3, "step_frac": bytes_ / secs / 1e9 / peak},
            "kernel_ms_per_step": {"restrict_plan": plan_ms / max(plan_n, 1),
                                   "restrict_rows": main_ms / max(main_n, 1),
                                   "restrict_final": fin_ms / max(fin_n, 1)},
            "clocks": clocks.summary(), "gpu_launches": 3 * args.steps, "device_status": status}
    print(json.dumps(line), flush=True)


def run_native(args, rank, world, local):
    import torch

    import speculative_decoding_token_gb300 as sv
    from speculative_decoding_token_gb300 import workload

    sv.build()
    cfg = workload.CONFIGS[args.config]
    batches = [workload.make_batch(args.config, device="cuda", seed=cfg["seed"] + 100 * rank + k)
               for k in range(args.batches)]
    B = cfg["B"]
    gm = batches[0].gamma_max
    h = sv.SpecVerify(B, gm, cfg["V"])
    stream = torch.cuda.current_stream()
    n_out = torch.empty(B, dtype=torch.int32, device="cuda")
    t_out = torch.empty(B, gm + 1, dtype=torch.int32, device="cuda")
    structs = [sv.make_batch_struct(b.target, b.draft, b.p_row_off, b.q_row_off,
                                    b.draft_tokens, b.gamma) for b in batches]

    greedy = args.mode == "greedy"

    lossy = args.mode == "lossy"

    def step(i):
        if greedy:
            sv.specverify_verify_greedy(h.h, structs[i % len(structs)], n_out, t_out,
                                        stream=stream)
        elif lossy:
            sv.specverify_verify_lossy(h.h, structs[i % len(structs)], cfg["T"],
                                       1_000_003 * (i + 1), "sq", 0.5, n_out, t_out,
                                       stream=stream)
        else:
            sv.specverify_verify(h.h, structs[i % len(structs)], cfg["T"], 1_000_003 * (i + 1),
                                 n_out, t_out, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # Which kernels a step launches (one more warm-up step, with the library's
    # per-kernel events). A sampling step is one launch (the fused kernel, or
    # the cluster kernel for a small batch): its kernel time is then the timed
    # region's time per step, and no per-kernel events are recorded in the
    # timed region (their two records a launch add about 4 us to a 17 us step).
    candidates = ((sv.KERNEL_PLAN, sv.KERNEL_ROWSTATS, sv.KERNEL_ACCEPT, sv.KERNEL_SMALL)
                  if greedy else (sv.KERNEL_FUSED, sv.KERNEL_SMALL))
    h.set_timing(True)
    h.get_timing(0, reset=True)
    step(args.warmup)
    torch.cuda.synchronize()
    launched = tuple(k for k in candidates if h.get_timing(k)[1] > 0)
    h.get_timing(0, reset=True)
    single = len(launched) == 1
    h.set_timing(not single)
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.25)
        start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        stop.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.05)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world)
    kernels = launched or candidates[:1]
    if single:
        per_kernel = {kernels[0]: (ms, args.steps)}
    else:
        per_kernel = {k: h.get_timing(k) for k in kernels}
    h.set_timing(False)
    status = h.device_status()

    timed = [batches[i % len(batches)] for i in range(args.warmup, args.warmup + args.steps)]
    tokens = sum(b.draft_token_count() for b in timed)
    logit_bytes = sum(b.logit_bytes(greedy=greedy) for b in timed)
    # The bytes each step needs: rows p_1..p_{n+1} and q_1..q_{min(n+1, gamma)}
    # of every sequence (rows after the first rejection cannot change the
    # result and are not read). n depends on the step's seed; the verify is
    # deterministic, so the timed steps are replayed untimed to read it.
    needed_bytes = 0
    # greedy: every target row is read once, and nothing else
    for i in (range(args.warmup, args.warmup + args.steps) if not greedy else ()):
        step(i)
        b = batches[i % len(batches)]
        n_h = n_out.cpu().long()
        g_h = b.gamma.cpu().long()
        rows = torch.where(n_h < g_h, 2 * (n_h + 1), 2 * g_h + 1)
        rows = torch.where(n_h < 0, torch.zeros_like(rows), rows)
        needed_bytes += int(rows.sum()) * b.V * b.target.element_size()
    if greedy:
        needed_bytes = logit_bytes
    secs = ms / 1e3
    value = job_throughput(world, tokens, secs)
    peak, peak_kind = peaks()
    # Dominant kernel: the fused sampling kernel (greedy: the row-statistics
    # kernel). Its algorithmic bytes are the per-call logit bytes of the
    # verify step -- every row of the batch read once, sum_b (2 gamma_b + 1)
    # V elem (greedy: the target rows) -- over its CUDA-event time. The bytes
    # the result needs (rows after a sequence's first rejection are not read)
    # give the stricter needed-bytes fraction; the ncu traffic, when its
    # stored capture matches these kernel sources, shows the re-reads.
    dom = sv.KERNEL_ROWSTATS if sv.KERNEL_ROWSTATS in kernels else kernels[0]
    k_ms, k_n = per_kernel[dom]
    k_avg = k_ms / max(k_n, 1)
    alg_bytes = logit_bytes / args.steps
    need_bytes = needed_bytes / args.steps
    achieved = alg_bytes / (k_avg / 1e3) / 1e9
    achieved_needed = need_bytes / (k_avg / 1e3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "fused_traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                tr = json.load(f)
            if (not greedy and tr.get("kernel_source_hash") == kernel_hash()
                    and tr.get("workload") == cfg["name"]):
                traffic = tr.get("traffic_bytes_per_launch")
        except Exception:
            traffic = None

    # end to end through the public API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        nb = len(batches)
        hb = [[t.cpu().pin_memory() if t is not None else None
               for t in (b.target, None if greedy else b.draft, b.p_row_off,
                         None if greedy else b.q_row_off, b.draft_tokens, b.gamma)]
              for b in batches]
        h2d = sum(t.numel() * t.element_size() for t in hb[0] if t is not None)
        d2h = B * 4 + B * (gm + 1) * 4
        for i in range(2):
            h.verify(*hb[i % nb], cfg["T"], 7 + i, greedy=greedy)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        e2e_tokens = 0
        for i in range(args.e2e_steps):
            h.verify(*hb[i % nb], cfg["T"], 11 + i, greedy=greedy)
            e2e_tokens += batches[i % nb].draft_token_count()
        torch.cuda.synchronize()
        e2e_secs = max_over_ranks(time.perf_counter() - t0, world)
        e2e = {"value": job_throughput(world, e2e_tokens, e2e_secs), "unit": UNIT,
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(batches[0], max(1, min(os.cpu_count() or 1, 64)), greedy)
    h.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(cfg, batches[0], args.mode),
        "hbm_gbs_per_gpu": logit_bytes / secs / 1e9,
        "hbm_frac_of_peak": logit_bytes / secs / 1e9 / peak,
        "needed_bytes_per_step": need_bytes,
        "needed_gbs": needed_bytes / secs / 1e9,
        "roofline": {"bound": "hbm",
                     "kernel": "rowstats_kernel" if dom == sv.KERNEL_ROWSTATS else
                     ("small_kernel" if dom == sv.KERNEL_SMALL else "fused_kernel"),
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "algorithmic_bytes": "sum_b (2 gamma_b + 1) V elem: every logit row of "
                                          "the step once" if not greedy else
                                          "sum_b (gamma_b + 1) V elem: every target row once",
                     "kernel_us": k_avg * 1e3,
                     "kernel_timing": "the timed region per step (one launch a step)" if single
                     else "per-kernel CUDA events on the launching stream",
                     "needed_bytes_per_launch": need_bytes,
                     "achieved_needed": achieved_needed, "frac_needed": achieved_needed / peak,
                     "step_achieved": alg_bytes / (ms / args.steps / 1e3) / 1e9,
                     "step_frac": alg_bytes / (ms / args.steps / 1e3) / 1e9 / peak,
                     "traffic_over_algorithmic": traffic / alg_bytes if traffic else None,
                     "traffic_over_needed": traffic / need_bytes if traffic else None},
        "kernel_ms_per_step": {{sv.KERNEL_PLAN: "plan", sv.KERNEL_ROWSTATS: "rowstats",
                                sv.KERNEL_ACCEPT: "accept", sv.KERNEL_FUSED: "fused",
                                sv.KERNEL_SMALL: "small"}[k]:
                               per_kernel[k][0] / max(per_kernel[k][1], 1) for k in kernels},
        "e2e": e2e,
        "cpu_baseline": cb,
        "clocks": clocks.summary(),
        "gpu_launches": len(kernels) * args.steps,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.mode in ("stats", "features"):
            run_diagnostics(args, rank, world, local)
        elif args.mode == "restricted":
            run_restricted(args, rank, world, local)
        else:
            run_native(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
