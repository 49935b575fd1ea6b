"""Throughput of the speculative-decoding verify/accept step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5] [--impl reference]

One step = one spec_verify call over one batch of the workload (config 3 adds
the MTP shift/insert with its hidden-state carry copy).  The default workload
is the largest one that fits one GPU, the large ragged batch: B=1024
requests, n_b ~ U{1..7} drafts, V=152064, bf16 logits, per-request T ~
U[0.3, 1.3].  Inputs rotate over enough replicas that the timed loop reads
more than four L2s' worth of distinct memory, so no step is served from L2.
Besides the timing, the CPU oracle (all host cores) checks every request of
the timed batch and the line reports its near-tie rows.

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(weak scaling, no collective on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified rows/s and tokens emitted/s at 1 GB300; achieved HBM GB/s vs 8 TB/s"
L2_BYTES = 129 * 2**20
NOMINAL_HBM_GBS = 8000.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "spec_verify_traffic.txt")


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_traffic(config_id, digest: str):
    """ncu DRAM bytes (read + write) per launch of the verify kernel recorded
    under profiles/ for this workload, if the kernel sources still hash to the
    digest recorded with them."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    rec = {}
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_digest") != digest:
        return None
    try:
        return float(rec[f"config{config_id}_dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    group = None
    if world > 1:
        import torch.distributed as dist

        backend = os.environ.get("SPECDEC_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
        group = dist.group.WORLD
    return rank, local, world, group


def aggregate(local_seconds: float, local_units: float, world: int, device="cpu"):
    """(max seconds over ranks, sum of units over ranks)."""
    if world <= 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ CPU oracle legs
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_call(inp, threads: int, want_margins: bool = False):
    """One oracle pass over the requests in `inp`, split into `threads`
    contiguous slices run side by side (the C oracle runs without the GIL).
    Request ids stay global, so the random draws are the whole batch's."""
    import concurrent.futures

    import numpy as np

    import oracle

    t, d, x, L, T, seed = inp
    n = len(L)
    parts = [p for p in np.array_split(np.arange(n), max(1, min(threads, n))) if len(p)]

    def run(p):
        sl = slice(p[0], p[-1] + 1)
        return oracle.spec_verify(t[sl], None if d is None else d[sl], x[sl], L[sl], T[sl], seed,
                                  req_ids=p.astype(np.int32), want_stats=want_margins)

    if len(parts) == 1:
        outs = [run(parts[0])]
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(parts)) as ex:
            outs = list(ex.map(run, parts))
    res = {k: np.concatenate([o[k] for o in outs], axis=0) for k in ("accepted_len", "out_tokens")}
    if want_margins:
        for k in ("accept_margin", "race_gap"):
            res[k] = np.concatenate([o[k] for o in outs], axis=0)
    return res


def host_inputs(w, nreq=None):
    from workloads.gen import logits_numpy

    nreq = w.B if nreq is None else min(w.B, nreq)
    t = logits_numpy(w.target[:nreq])
    d = None if w.draft is None else logits_numpy(w.draft[:nreq])
    x = w.draft_tokens[:nreq].cpu().numpy()
    L = w.draft_len[:nreq].cpu().numpy()
    T = w.temperature[:nreq].cpu().numpy()
    return (t, d, x, L, T, w.seed)


def oracle_sample_rate(w, budget_s: float, max_requests: int = None, threads: int = 1):
    """Oracle rows/s on the host: whole requests of `w` (copied to the host),
    repeated until `budget_s` of CPU time has been spent, on `threads` host
    threads (slices of the requests side by side)."""
    import oracle

    inp = host_inputs(w, max_requests)
    L = inp[3]
    rows_per_call = int((L + 1).sum())
    oracle.lib()
    calls, t0 = 0, time.perf_counter()
    while True:
        r = oracle_call(inp, threads)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    tokens = int((r["accepted_len"] + 1).sum()) * calls
    return {"rows_per_s": rows_per_call * calls / el, "tokens_per_s": tokens / el, "seconds": el,
            "calls": calls, "requests": len(L), "rows_per_call": rows_per_call, "threads": threads}


def oracle_parity(w, acc, out, threads: int):
    """Every request of the timed batch against the oracle: requests that
    differ, and the rows whose decision margin is below 1e-5 (near ties,
    where fp32 and fp64 may decide differently)."""
    import numpy as np

    NEAR = 1e-5
    ref = oracle_call(host_inputs(w), threads, want_margins=True)
    a = acc.cpu().numpy()
    o = out.cpu().numpy().reshape(ref["out_tokens"].shape)
    near = np.zeros(len(a), dtype=np.int64)
    for i in range(len(a)):
        m = ref["accept_margin"][i]
        m = m[~np.isnan(m)]
        g = ref["race_gap"][i]
        near[i] = int((m < NEAR).sum()) + int(np.isfinite(g) and g < NEAR)
    mism = (a != ref["accepted_len"]) | (o != ref["out_tokens"]).any(axis=1)
    return {"requests": int(len(a)), "rows": int((w.draft_len.cpu().numpy().clip(0, w.n_max) + 1).sum()),
            "mismatched_requests": int(mism.sum()), "mismatched_without_near_tie": int((mism & (near == 0)).sum()),
            "near_tie_rows": int(near.sum()), "oracle_threads": threads}


def run_reference(args):
    """The oracle as it stands, timed on the host cores: each step is one
    oracle call over a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import torch

    import oracle
    from workloads import make_config
    from workloads.gen import logits_numpy

    cores = host_cores()
    nreq = args.ref_requests or cores
    w = make_config(args.config, device="cpu", B=nreq)  # same recipe, a bounded sample
    inp = host_inputs(w, nreq)
    nreq = len(inp[3])
    rows = int((inp[3] + 1).sum())
    oracle.lib()
    for _ in range(args.warmup):
        oracle_call(inp, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_call(inp, cores)
    el = time.perf_counter() - t0
    tokens = int((r["accepted_len"] + 1).sum())
    value = rows * args.steps / el
    sample = (f"{nreq} requests ({rows} target rows) of the workload's recipe per step, "
              f"fp64 C oracle on {cores} host threads (slices of the requests side by side)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_emitted_per_s": tokens * args.steps / el,
        "config": {"workload": w.name, "B": w.B, "n": w.n_max, "V": w.V, "sampled_requests": nreq},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def shard_cuts(V: int, S: int):
    """Vocabulary boundaries of S shards, as even as 8-element steps allow."""
    step = -(-V // (8 * S)) * 8
    return [0] + [min(V, step * s) for s in range(1, S)] + [V]


def run_gpu(args):
    import numpy as np
    import torch

    import speculative_decoding_verification_80_gb300 as sd
    from speculative_decoding_verification_80_gb300 import build as sd_build
    from workloads import make_config
    from workloads.gen import algorithmic_bytes

    rank, local, world, _ = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sd.load_library()

    w = make_config(args.config, device=dev, B=args.batch)
    B, n, V = w.B, w.n_max, w.V
    rows_t, rows_d = w.rows_target, w.rows_draft
    alg_bytes = algorithmic_bytes(w)
    S = args.shards
    cuts = shard_cuts(V, S)
    if args.packed:
        from workloads import pack

        pt, pd, ptok, cu = pack(w)
        base = (pt, pd)
    elif S > 1:  # each shard holds the vocabulary range [cuts[s], cuts[s+1]) of every row
        base = ([w.target[..., cuts[s]:cuts[s + 1]].contiguous() for s in range(S)],
                None if w.draft is None else [w.draft[..., cuts[s]:cuts[s + 1]].contiguous() for s in range(S)])
    else:
        base = (w.target, w.draft)

    def nbytes(x):
        if x is None:
            return 0
        return sum(t.numel() * t.element_size() for t in x) if isinstance(x, list) else x.numel() * x.element_size()

    def clone(x):
        if x is None:
            return None
        return [t.clone() for t in x] if isinstance(x, list) else x.clone()

    in_bytes = nbytes(base[0]) + nbytes(base[1])
    reps = max(2, math.ceil(4 * L2_BYTES / max(1, in_bytes)))
    replicas = [base] + [(clone(base[0]), clone(base[1])) for _ in range(reps - 1)]
    exch = sd.shard_exchange_buffers(S, B, n, device=dev) if S > 1 else None
    ws = sd.new_workspace(B, n, V, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, n + 1, dtype=torch.int32, device=dev)
    mtp = args.config == 3
    if mtp:
        tok_out = torch.empty_like(w.mtp_tokens)
        hid_out = torch.empty_like(w.hidden)
    stream = torch.cuda.Stream(device=dev)

    if args.packed:
        out = torch.empty(pt.shape[0], dtype=torch.int32, device=dev)

    def step(i):
        tgt, drf = replicas[i % reps]
        if args.packed:
            sd.spec_verify_packed(tgt, drf, cu, ptok, w.temperature, n, seed=w.seed, accepted_len=acc,
                                  out_tokens=out, workspace=ws, stream=stream)
        elif args.early_exit:
            sd.spec_verify_early_exit(tgt, drf, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                      accepted_len=acc, out_tokens=out, workspace=ws, stream=stream)
        elif S > 1:
            sd.spec_verify_sharded(tgt, drf, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                   accepted_len=acc, out_tokens=out, exchange=exch, stream=stream)
        else:
            sd.spec_verify(tgt, drf, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                           accepted_len=acc, out_tokens=out, workspace=ws, stream=stream)
        if mtp:
            sd.mtp_shift_insert(w.mtp_tokens, tok_out, w.draft_len, acc, out.view(-1), n + 1,
                                hidden_in=w.hidden, hidden_out=hid_out, stream=stream)

    # CUDA graphs, one per replica, each capturing G consecutive steps (one
    # kernel launch per step, each on its own replica), so host and graph
    # launch costs stay off the clock; G divides K so exactly K steps run.
    K = args.steps
    G = max(q for q in range(1, max(1, args.graph_steps) + 1) if K % q == 0)
    graphs = []
    with torch.cuda.stream(stream):
        for i in range(2):
            step(i)
    torch.cuda.synchronize(dev)
    for r in range(reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for q in range(G):
                step(r + q)
        graphs.append(g)
    torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for i in range(-(-args.warmup // G)):
            graphs[i % reps].replay()
    torch.cuda.synchronize(dev)

    KR = K // G  # graph replays in the timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(KR)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    if args.early_exit:
        sd.bytes_read(ws)  # count only the timed steps
    with ClockSampler(local) as clocks:
        time.sleep(0.25)  # let the sampler start before the loop
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(KR):
                ev[i][0].record(stream)
                graphs[i % reps].replay()
                ev[i][1].record(stream)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kernel_s = statistics.mean(step_ms[len(step_ms) // 10:] or step_ms) / 1e3 / G  # per launch
    emitted = int((acc.to(torch.int64) + 1).sum().item())
    seconds, total_rows = aggregate(elapsed, rows_t * K, world)
    _, total_tokens = aggregate(elapsed, emitted * K, world)
    peak, peak_kind = measured_peaks()

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(w, sd, dev, stream, args, packed=(pt, pd, ptok, cu) if args.packed else None, cuts=cuts)
    cpu = cpu1 = parity = None
    if rank == 0 and not args.no_cpu_baseline:
        cores = host_cores()
        cpu_w = make_config(args.config, device="cpu", B=min(B, max(args.cpu_requests, cores)))
        r = oracle_sample_rate(cpu_w, args.cpu_seconds, threads=cores)
        cpu = {"value": r["rows_per_s"], "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"{r['requests']} requests ({r['rows_per_call']} target rows) of the "
                         f"workload's recipe, repeated {r['calls']}x over {r['seconds']:.1f} s, "
                         f"fp64 C oracle on {cores} host threads (slices of the requests side by side)"}
        r1 = oracle_sample_rate(cpu_w, args.cpu_seconds / 3, max_requests=min(8, cpu_w.B), threads=1)
        cpu1 = {"value": r1["rows_per_s"], "unit": "rows/s", "cores": 1, "kind": "oracle",
                "sample": f"{r1['requests']} requests ({r1['rows_per_call']} target rows), repeated "
                          f"{r1['calls']}x over {r1['seconds']:.1f} s, 1 thread"}
        if not (args.packed or S > 1):
            parity = oracle_parity(w, acc, out, cores)
    if rank != 0:
        return 0
    ee = None
    if args.early_exit:
        # The method needs target rows 0..a_b and draft rows 0..min(a_b, n_b - 1)
        # of sampled requests; the kernel reports what it actually read.
        a = acc.cpu().numpy().astype(np.int64)
        L = w.draft_len.cpu().numpy().clip(0, n).astype(np.int64)
        sampled = (w.temperature.cpu().numpy() > 0) & (w.draft is not None)
        row_b = V * w.target.element_size()
        need = int(((a + 1) + np.where(sampled, np.minimum(a + 1, L), 0)).sum() * row_b)
        ee = {"needed_bytes_per_step": need, "bytes_read_per_step": sd.bytes_read(ws) / K,
              "full_rows_bytes_per_step": alg_bytes}
        alg_bytes = need
    achieved = alg_bytes / kernel_s / 1e9
    digest = sd_build.verify_digest()
    line = {
        "metric": METRIC, "value": total_rows / seconds, "unit": "rows/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": seconds / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "accumulate": "f32", "data": "synthetic",
        "tokens_emitted_per_s": total_tokens / seconds,
        "hbm_gbs_algorithmic": alg_bytes * K * world / seconds / 1e9,
        "frac_of_8tbs": alg_bytes * K * world / seconds / 1e9 / NOMINAL_HBM_GBS,
        "config": {"workload": w.name + (" packed" if args.packed else "") + (" early-exit" if args.early_exit else "")
                   + (f" vocab-sharded S={S}" if S > 1 else ""),
                   "B": B, "n": n, "V": V,
                   "logits": w.dtype, "layout": "packed rows (cu_rows)" if args.packed else (
                       f"dense [B, n+1, V] split into {S} vocabulary shards at {cuts[1:-1]}" if S > 1
                       else "dense [B, n+1, V]"),
                   "target_rows": rows_t, "draft_rows": rows_d,
                   "algorithmic_bytes_per_step": alg_bytes,
                   "l2": f"inputs rotate over {reps} replicas ({reps * in_bytes / 2**20:.0f} MiB "
                         f"> 4x the 129 MB L2)",
                   "timing": f"CUDA events on the launch stream; one CUDA graph replay per {G} steps "
                             "(one kernel launch per step, each on its own input replica)",
                   "mean_emitted_per_request": emitted / B},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "traffic": read_traffic(f"{args.config}{'_packed' if args.packed else ''}"
                                             f"{'_early_exit' if args.early_exit else ''}"
                                             f"{f'_shards{S}' if S > 1 else ''}", digest),
                     "kernel": (f"shard_stats_kernel x{S} + shard_race_kernel x{S} + shard_finish_kernel "
                                "(the whole step)") if S > 1 else "verify_persistent_kernel",
                     "kernel_avg_us": kernel_s * 1e6,
                     "source_digest": digest},
        **({"early_exit": ee} if ee else {}),
        "cpu_baseline": cpu,
        "cpu_baseline_1_thread": cpu1,
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": K * ((2 * S + 1 if S > 1 else 1) + (1 if mtp else 0)),
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(w, sd, dev, stream, args, packed=None, cuts=None):
    """Same metric through the public call with host inputs: each step copies
    that step's inputs from pinned host memory, verifies, and reads the
    results back."""
    import torch

    S = len(cuts) - 1 if cuts is not None else 1
    if packed is None and S > 1:  # one host buffer per vocabulary shard
        host = {k: getattr(w, k).cpu().pin_memory() for k in ("draft_tokens", "draft_len", "temperature")}
        for s in range(S):
            host[f"target{s}"] = w.target[..., cuts[s]:cuts[s + 1]].contiguous().cpu().pin_memory()
            if w.draft is not None:
                host[f"draft{s}"] = w.draft[..., cuts[s]:cuts[s + 1]].contiguous().cpu().pin_memory()
        out_shape = (w.B, w.n_max + 1)
    elif packed is None:
        host = {k: getattr(w, k).cpu().pin_memory() for k in
                ("target", "draft", "draft_tokens", "draft_len", "temperature") if getattr(w, k) is not None}
        out_shape = (w.B, w.n_max + 1)
    else:  # packed rows: only the valid rows cross the link
        pt, pd, ptok, cu = packed
        host = {"target": pt.cpu().pin_memory(), "draft_tokens": ptok.cpu().pin_memory(),
                "cu_rows": cu.cpu().pin_memory(), "temperature": w.temperature.cpu().pin_memory()}
        if pd is not None:
            host["draft"] = pd.cpu().pin_memory()
        out_shape = (pt.shape[0],)
    devb = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    acc_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
    out_h = torch.empty(out_shape, dtype=torch.int32).pin_memory()
    acc = torch.empty(w.B, dtype=torch.int32, device=dev)
    out = torch.empty(out_shape, dtype=torch.int32, device=dev)
    ws = sd.new_workspace(w.B, w.n_max, w.V, device=dev)
    exch = sd.shard_exchange_buffers(S, w.B, w.n_max, device=dev) if S > 1 else None
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = acc_h.numel() * 4 + out_h.numel() * 4

    def one():
        with torch.cuda.stream(stream):
            for k, v in host.items():
                devb[k].copy_(v, non_blocking=True)
            if packed is None and S > 1:
                sd.spec_verify_sharded([devb[f"target{s}"] for s in range(S)],
                                       [devb[f"draft{s}"] for s in range(S)] if w.draft is not None else None,
                                       devb["draft_tokens"], devb["draft_len"], devb["temperature"], seed=w.seed,
                                       accepted_len=acc, out_tokens=out, exchange=exch, stream=stream)
            elif packed is None and args.early_exit:
                sd.spec_verify_early_exit(devb["target"], devb.get("draft"), devb["draft_tokens"],
                                          devb["draft_len"], devb["temperature"], seed=w.seed, accepted_len=acc,
                                          out_tokens=out, workspace=ws, stream=stream)
            elif packed is None:
                sd.spec_verify(devb["target"], devb.get("draft"), devb["draft_tokens"],
                               devb["draft_len"], devb["temperature"], seed=w.seed, accepted_len=acc,
                               out_tokens=out, workspace=ws, stream=stream)
            else:
                sd.spec_verify_packed(devb["target"], devb.get("draft"), devb["cu_rows"], devb["draft_tokens"],
                                      devb["temperature"], w.n_max, seed=w.seed, accepted_len=acc,
                                      out_tokens=out, workspace=ws, stream=stream)
            acc_h.copy_(acc, non_blocking=True)
            out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    steps = max(3, args.e2e_steps)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    sec = a.elapsed_time(b) / 1e3
    return {"value": w.rows_target * steps / sec, "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": sec / steps * 1e3}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-requests", type=int, default=8,
                    help="requests in the CPU baseline's sample (at least one per host core)")
    ap.add_argument("--ref-requests", type=int, default=0,
                    help="requests per step of the reference arm (default: one per host core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph-steps", type=int, default=8,
                    help="steps captured per CUDA graph replay (the largest divisor of --steps up to this)")
    ap.add_argument("--early-exit", action="store_true",
                    help="time spec_verify_early_exit (rows after a request's first rejection are not read)")
    ap.add_argument("--packed", action="store_true",
                    help="time spec_verify_packed on the workload's packed rows instead of the dense call")
    ap.add_argument("--shards", type=int, default=1,
                    help="time the vocabulary-sharded step with S shards on this GPU (dense layout)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's request count (same recipe); not the headline line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.packed and args.early_exit:
        ap.error("--packed and --early-exit are separate calls")
    if args.shards < 1 or (args.shards > 1 and (args.packed or args.early_exit or args.config == 3)):
        ap.error("--shards S (S >= 1) times the dense sharded call alone (not with --packed, --early-exit "
                 "or the MTP workload)")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
