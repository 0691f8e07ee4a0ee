#!/usr/bin/env python
"""Throughput of exact attention forward + backward on GB300.

One step = the whole hot path on one batch: fa_fwd (O, LSE) then fa_bwd
(preprocess, main loop, dQ conversion) on the causal d=128 workload
B=4, H=16, Nq=Nk=4096 (bf16, seeded N(0,1) inputs). The metric is TFLOP/s with
the convention forward = 4*B*H*Nq*Nk*d, backward = 2.5 x forward, both halved
for causal.

Prints ONE JSON line (rank 0). Under torchrun every rank runs its own replica
of the workload on its own GPU (different seed) with no data exchange; the
process group is used only for the barrier and the max-over-ranks timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
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
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

WORKLOAD = "bf16_b4h16_n4096_d128_causal_bwd"
FWD_EXTRA = "bf16_b2h32_n8192_d128_causal"
DECODE_EXTRA = "bf16_b8h32_q1_k32768_d128_decode"
METRIC = "attention fwd/bwd TFLOP/s (bf16, causal, d=128) and % of GB300 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# NVIDIA's nominal dense (no 2:4 sparsity) bf16 tensor rate of one GB300, for
# context beside the measured peaks
NOMINAL_BF16_TFLOPS = 2250.0


def flops(w):
    f = 4.0 * w.B * w.H * w.Nq * w.Nk * w.d * (0.5 if w.causal else 1.0)
    return f, (2.5 * f if w.backward else 0.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.15)
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
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def oracle_sample(w, n_rows_total, seed_offset=0):
    """Time the fp64 oracle on a bounded sample of workload w: `n_rows_total`
    query rows spread over as many heads as there are oracle threads, each
    head's rows processed on its own thread (forward rows, then their full
    backward contributions). Returns (seconds, conventional flops, description)."""
    import concurrent.futures

    import numpy as np
    import torch

    import oracle

    cores = oracle.num_threads()
    per_thread = max(1, n_rows_total // max(1, min(cores, w.B * w.H)))
    rows_per_head = min(w.Nq, per_thread)
    n_heads = max(1, min(w.B * w.H, -(-n_rows_total // rows_per_head)))
    key = (w.name, n_heads)
    if key not in _ORACLE_INPUTS:
        x = workloads.make_inputs(w.with_(B=1, H=n_heads), seed=w.seed + 777, with_dO=True)
        heads = []
        for h in range(n_heads):
            f = lambda t: np.ascontiguousarray(t[0, h].to(torch.float64).numpy())
            heads.append((f(x["q"]), f(x["k"]), f(x["v"]), f(x["dO"])))
        bias = None if x["bias"] is None else np.ascontiguousarray(x["bias"][0].double().numpy())
        _ORACLE_INPUTS[key] = (heads, bias)
    heads, bias = _ORACLE_INPUTS[key]
    rng = np.random.default_rng(seed_offset)
    rows = [np.sort(rng.choice(w.Nq, size=min(rows_per_head, w.Nq), replace=False))
            for _ in range(n_heads)]
    # conventional flops of the sampled rows: 4*vis*d forward + 10*vis*d backward
    conv = 0.0
    for r in rows:
        if w.causal:
            vis = np.minimum(r + (w.Nk - w.Nq) + 1, w.Nk).clip(min=0)
        else:
            vis = np.full(r.shape, w.Nk)
        conv += float(vis.sum()) * w.d * (4.0 + (10.0 if w.backward else 0.0))

    def work(h):
        qh, kh, vh, dOh = heads[h]
        oracle.fwd_head_rows(qh, kh, vh, bias, rows[h], w.scale, w.causal)
        if w.backward:
            oracle.bwd_head_rows(qh, kh, vh, bias, dOh, rows[h], w.scale, w.causal)

    threads = max(1, min(cores, n_heads))
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, range(n_heads)))
    dt = time.perf_counter() - t0
    desc = ("%d query rows (%d per head) of %d heads of %s: forward rows + their full "
            "backward contributions, fp64, one thread per head, %d threads" %
            (sum(len(r) for r in rows), len(rows[0]), n_heads, w.name, threads))
    return dt, conv, desc, threads


def calibrated_oracle(w, budget_s, seed_offset=0):
    """Pick a sample size so that one oracle sample takes about budget_s seconds."""
    import oracle
    cores = oracle.num_threads()
    probe = 16
    dt, conv, _, nh = oracle_sample(w, probe * max(1, min(cores, w.B * w.H)), seed_offset)
    per_row = dt / probe          # seconds per row on one head-thread (heads run in parallel)
    return int(max(1.0, budget_s / max(per_row, 1e-6))) * nh


def cpu_baseline(w, budget_s=12.0):
    n_rows = calibrated_oracle(w, budget_s / 4)
    dt, conv, desc, nh = oracle_sample(w, n_rows)
    for i in range(3):   # grow the sample until it takes about budget_s
        if dt >= 0.6 * budget_s or n_rows >= w.B * w.H * w.Nq:
            break
        n_rows = max(nh, int(n_rows * min(8.0, budget_s / max(dt, 1e-3))))
        dt, conv, desc, nh = oracle_sample(w, n_rows, seed_offset=1 + i)
    out = {"value": conv / dt / 1e12, "unit": UNIT, "cores": nh, "kind": "oracle",
           "sample": desc, "seconds": round(dt, 3)}
    out.update(one_thread_head(w))
    return out


def one_thread_head(w, n_rows=256):
    """The oracle on ONE thread for `n_rows` evenly spaced query rows of one head
    (forward rows + their full backward contributions), extrapolated to the whole
    head by the conventional FLOP count of the sampled vs all rows."""
    import numpy as np
    import torch

    import oracle

    x = workloads.make_inputs(w.with_(B=1, H=1), seed=w.seed + 778, with_dO=True)
    f = lambda t: np.ascontiguousarray(t[0, 0].to(torch.float64).numpy())
    qh, kh, vh, dOh = f(x["q"]), f(x["k"]), f(x["v"]), f(x["dO"])
    bias = None if x["bias"] is None else np.ascontiguousarray(x["bias"][0].double().numpy())
    rows = np.unique(np.linspace(0, w.Nq - 1, min(n_rows, w.Nq)).round().astype(np.int64))

    def visible(r):
        if w.causal:
            return np.minimum(r + (w.Nk - w.Nq) + 1, w.Nk).clip(min=0).astype(np.float64)
        return np.full(r.shape, float(w.Nk))
    t0 = time.perf_counter()
    oracle.fwd_head_rows(qh, kh, vh, bias, rows, w.scale, w.causal)
    if w.backward:
        oracle.bwd_head_rows(qh, kh, vh, bias, dOh, rows, w.scale, w.causal)
    dt = time.perf_counter() - t0
    frac = float(visible(rows).sum()) / float(visible(np.arange(w.Nq)).sum())
    return {"one_thread_head_seconds_extrapolated": round(dt / frac, 3),
            "one_thread_head_sample": "%d of %d query rows of one head on one thread "
                                      "(%.3f s), scaled by their share of the head's FLOPs"
                                      % (len(rows), w.Nq, dt)}


def bench_config(w, world):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
            "causal": w.causal, "step": "fa_fwd + fa_bwd",
            "flop_convention": "fwd 4*B*H*Nq*Nk*d, bwd 2.5x fwd, halved for causal",
            "l2": "inputs larger than L2 (q,k,v,dO 64 MiB each + outputs), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[WORKLOAD]
    total_budget = 150.0
    per_step = max(0.5, total_budget / max(1, args.steps + args.warmup))
    n_rows = calibrated_oracle(w, per_step)
    dt, _, _, _ = oracle_sample(w, n_rows)
    n_rows = max(1, int(n_rows * per_step / max(dt, 1e-3)))
    for i in range(args.warmup):
        oracle_sample(w, n_rows, seed_offset=i)
    times, convs = [], []
    desc = ""
    nh = 1
    for i in range(args.steps):
        dt, conv, desc, nh = oracle_sample(w, n_rows, seed_offset=100 + i)
        times.append(dt)
        convs.append(conv)
    value = sum(convs) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nh, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm

def replica_seed(w, rank):
    """Each replica draws its own batch: the workload's seed offset by the rank."""
    return w.seed + rank


def replica_throughput(ms_total_local, steps, flops_per_step, world, device=None):
    """Whole-job throughput of `world` independent replicas.

    The timed region of each rank is `ms_total_local` milliseconds for `steps`
    steps of `flops_per_step` FLOPs; the job time is the slowest rank's (MAX
    over ranks), and the job's work is every rank's. Returns (ms per step,
    TFLOP/s). With world > 1 this is a collective: every rank must call it.
    """
    import torch
    t = torch.tensor([float(ms_total_local)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_step = float(t.item()) / steps
    return ms_step, flops_per_step * world / (ms_step * 1e-3) / 1e12

def l2_flush_buffer(dev):
    """A 256 MiB buffer (about twice the 129 MB L2); writing it between timed
    launches evicts the previous launch's inputs and outputs from L2."""
    import torch
    return torch.empty(256 << 20, dtype=torch.uint8, device=dev)


def time_launches(fn, stream, flush, iters=10, warmup=3):
    """Median milliseconds of fn() over `iters` launches, each bracketed by its
    own CUDA events on `stream`, with L2 flushed (outside the events) before
    each one."""
    import torch
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    stream.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def effective_fwd_flops(w, key_len):
    """Forward FLOPs over the keys that are not masked: 4*H*Nq*d per valid key
    (key padding: L_b valid keys in batch b), halved for causal."""
    valid = float(sum(int(x) for x in key_len)) if key_len is not None else float(w.B * w.Nk)
    return 4.0 * w.H * w.Nq * valid * w.d * (0.5 if w.causal else 1.0)


def measure_configs(fa, dev, stream, rank, headline_parts):
    """Every workload the hot path is specified on, timed per launch with L2
    flushed between launches: throughput at the FLOP convention and as a
    fraction of the measured burst bf16 peak. Inputs are N(0,1) drawn on the
    device (a seeded device generator); the key-padding lengths are drawn on
    the host with the recipe of workloads.make_inputs."""
    import torch
    peaks, _ = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    flush = l2_flush_buffer(dev)
    out = {}

    def rec(ms, fl, eff=None):
        r = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_of_burst_peak":
             fl / (ms * 1e-3) / 1e12 / peak}
        if eff is not None:
            # key padding: the masked key tiles are skipped, so the fraction
            # of the peak that means anything is the one on valid keys
            r["effective_tflops"] = eff / (ms * 1e-3) / 1e12
            r["effective_frac_of_burst_peak"] = eff / (ms * 1e-3) / 1e12 / peak
        return r

    for name in ("f32_b1h1_n128_d64", "bf16_b4h16_n2048_d64", "bf16_b2h32_n8192_d128_causal",
                 "bf16_b4h16_n4096_d128_causal_bwd", "bf16_b8h16_q1024_k16384_d128_keypad"):
        w = workloads.WORKLOADS[name]
        g = torch.Generator(device=dev).manual_seed(w.seed + 31 * rank)
        dt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
        q, dO = (torch.randn((w.B, w.H, w.Nq, w.d), generator=g, device=dev, dtype=dt)
                 for _ in range(2))
        k, v = (torch.randn((w.B, w.H, w.Nk, w.d), generator=g, device=dev, dtype=dt)
                for _ in range(2))
        bias, key_len = None, None
        if w.key_padding:
            gh = torch.Generator().manual_seed(w.seed + 31 * rank)
            key_len = torch.randint(w.Nk // 2, w.Nk + 1, (w.B,), generator=gh).tolist()
            bias = torch.zeros((w.B, w.Nk), dtype=torch.float32)
            for b, L in enumerate(key_len):
                bias[b, L:] = float("-inf")
            bias = bias.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
        for causal in ((False, True) if name == "bf16_b4h16_n2048_d64" else (w.causal,)):
            wc = w.with_(causal=causal)
            kw = dict(key_bias=bias, causal=causal, scale=w.scale)
            key = name + ("_causal" if causal and "causal" not in name else "")
            f_fwd = flops(wc)[0]
            ms = time_launches(lambda: fa.fwd(q, k, v, out=o, lse=lse, **kw), stream, flush)
            if w.dtype == "fp32":
                out[key] = {"fwd": {"us": ms * 1e3}}
                continue
            ent = {"fwd": rec(ms, f_fwd, effective_fwd_flops(wc, key_len) if bias is not None
                              else None)}
            if name != "bf16_b2h32_n8192_d128_causal":
                ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d),
                                 dtype=torch.uint8, device=dev)
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                fa.fwd(q, k, v, out=o, lse=lse, **kw)
                bk = dict(workspace=ws, dq=dq, dk=dk, dv=dv, **kw)
                ms_b = time_launches(lambda: fa.bwd(q, k, v, o, lse, dO, **bk), stream, flush)
                # the main launch alone (after one preprocess; repeating it only
                # adds more into the dQ accumulator, the work is the same)
                fa.bwd(q, k, v, o, lse, dO, stage="preprocess", **bk)
                ms_m = time_launches(lambda: fa.bwd(q, k, v, o, lse, dO, stage="main", **bk),
                                     stream, flush)
                eff_b = (2.5 * effective_fwd_flops(wc, key_len) if bias is not None else None)
                ent["bwd"] = rec(ms_b, 2.5 * f_fwd, eff_b)
                ent["bwd_main"] = rec(ms_m, 2.5 * f_fwd, eff_b)
                del ws, dq, dk, dv
            if name == WORKLOAD:
                ent["in_step_ms_median"] = {n: statistics.median(v_)
                                            for n, v_ in headline_parts.items()}
            out[key] = ent
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        del q, k, v, dO, o, lse, bias
    del flush
    out["timing"] = ("per launch, CUDA events on the launching stream, median of 10 after 3 "
                     "warm-ups, L2 flushed (256 MiB write) before each launch; FLOPs: forward "
                     "4*B*H*Nq*Nk*d, backward 2.5x, halved for causal; key padding: nominal "
                     "(all Nk keys) and effective (valid keys only) counts")
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import exact_io_aware_03_gb300 as fa
    from exact_io_aware_03_gb300 import build as fa_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        fa_build.build()
    if world > 1:
        dist.barrier()
    fa.load()

    w = workloads.WORKLOADS[WORKLOAD]
    f_fwd, f_bwd = flops(w)
    x = workloads.make_inputs(w, with_dO=True, seed=replica_seed(w, rank))
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(causal=w.causal, scale=w.scale)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fwd(q, k, v, out=o, lse=lse, **kw)
        if ev is not None:
            ev[1].record(stream)
        fa.bwd(q, k, v, o, lse, dO, workspace=ws, dq=dq, dk=dk, dv=dv, stage="preprocess", **kw)
        if ev is not None:
            ev[2].record(stream)
        fa.bwd(q, k, v, o, lse, dO, workspace=ws, dq=dq, dk=dk, dv=dv, stage="main", **kw)
        if ev is not None:
            ev[3].record(stream)
        fa.bwd(q, k, v, o, lse, dO, workspace=ws, dq=dq, dk=dk, dv=dv, stage="postprocess", **kw)
        if ev is not None:
            ev[4].record(stream)

    launches_per_step = 4   # fwd, bwd preprocess, bwd main, bwd postprocess
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    fa.check_device_error(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    fa.check_device_error(dev)
    ms_total = t_start.elapsed_time(t_end)
    parts = {n: [e[j].elapsed_time(e[j + 1]) for e in evs]
             for j, n in enumerate(["fwd", "bwd_preprocess", "bwd_main", "bwd_postprocess"])}
    ms_step, value = replica_throughput(ms_total, args.steps, f_fwd + f_bwd, world, dev)

    # ---- end to end through the public API: every step uploads its inputs
    # from pinned host memory, runs fa_fwd + fa_bwd and downloads all of its
    # results (O, LSE, dQ, dK, dV). Steps are pipelined the way a training
    # loop would run them: three streams (upload step k+1 / compute step k /
    # download step k-1) over two sets of device and host buffers, ordered
    # by events; the timed region runs from the first upload to the last
    # download.
    e2e_steps = max(4, min(args.steps, 20))
    names_in, names_out = ("q", "k", "v", "dO"), ("o", "lse", "dq", "dk", "dv")
    host_in = {n: x[n].pin_memory() for n in names_in}
    dev_in = [{"q": q, "k": k, "v": v, "dO": dO},
              {n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO))}]
    dev_out = [{"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
               {n: torch.empty_like(t) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                   ("dv", dv))}]
    host_out = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in dev_out[0].items()}
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    # one copy stream per direction (spreading the copies over more streams
    # measured slower: the host link, not the copy engines, limits them)
    NC = 1
    s_comp = torch.cuda.Stream(dev)
    s_ups = [torch.cuda.Stream(dev) for _ in range(NC)]
    s_downs = [torch.cuda.Stream(dev) for _ in range(NC)]
    s_up, s_down = s_ups[0], s_downs[0]
    ev_up = [[torch.cuda.Event() for _ in range(NC)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [[torch.cuda.Event() for _ in range(NC)] for _ in range(2)]

    def e2e_run(steps, t0=None, t1=None):
        for j in range(2):   # nothing outstanding on either buffer set
            ev_comp[j].record(stream)
            for e in ev_up[j] + ev_down[j]:
                e.record(stream)
        for s_ in [s_comp] + s_ups + s_downs:
            s_.wait_stream(stream)
        if t0 is not None:
            t0.record(stream)
        for i in range(steps):
            j = i % 2
            di, do_, ho = dev_in[j], dev_out[j], host_out[j]
            for c, n in enumerate(names_in):
                su = s_ups[c % NC]
                su.wait_event(ev_comp[j])        # step i-2 has read these inputs
                with torch.cuda.stream(su):
                    di[n].copy_(host_in[n], non_blocking=True)
            for c in range(NC):
                ev_up[j][c].record(s_ups[c])
                s_comp.wait_event(ev_up[j][c])
                s_comp.wait_event(ev_down[j][c])   # step i-2's results have left
            with torch.cuda.stream(s_comp):
                fa.fwd(di["q"], di["k"], di["v"], out=do_["o"], lse=do_["lse"], **kw)
                fa.bwd(di["q"], di["k"], di["v"], do_["o"], do_["lse"], di["dO"], workspace=ws,
                       dq=do_["dq"], dk=do_["dk"], dv=do_["dv"], **kw)
                ev_comp[j].record(s_comp)
            for c, n in enumerate(names_out):
                sd = s_downs[c % NC]
                sd.wait_event(ev_comp[j])
                with torch.cuda.stream(sd):
                    ho[n].copy_(do_[n], non_blocking=True)
            for c in range(NC):
                ev_down[j][c].record(s_downs[c])
        if t1 is not None:
            for s_ in [s_comp] + s_ups + s_downs:
                stream.wait_stream(s_)
            t1.record(stream)
        torch.cuda.synchronize(dev)

    e2e_run(2)
    if world > 1:
        dist.barrier()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, a0, a1)
    fa.check_device_error(dev)
    _, e2e_value = replica_throughput(a0.elapsed_time(a1), e2e_steps, f_fwd + f_bwd, world, dev)
    del dev_in[1], dev_out[1]

    # ---- extra forward-only measurement on the long-context causal workload
    extras = {}
    if not args.no_extras:
        we = workloads.WORKLOADS[FWD_EXTRA]
        g = torch.Generator(device=dev).manual_seed(we.seed + rank)
        extras["configs"] = measure_configs(fa, dev, stream, rank, parts)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e = 20
        # decode step through the split-KV forward: HBM-bound (K and V read once)
        wd = workloads.WORKLOADS[DECODE_EXTRA]
        qd, kd, vd = (torch.randn((wd.B, wd.H, n, wd.d), generator=g, device=dev,
                                  dtype=torch.bfloat16) for n in (wd.Nq, wd.Nk, wd.Nk))
        with torch.cuda.device(dev):
            ns = fa.fa_fwd_splitkv_default_splits(wd.B, wd.H, wd.Nq, wd.Nk, wd.d)
        wsd = torch.empty(fa.fa_fwd_splitkv_workspace_size(wd.B, wd.H, wd.Nq, wd.Nk, wd.d, ns),
                          dtype=torch.uint8, device=dev)
        od = torch.empty_like(qd)
        ld = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(3):
            fa.fwd_splitkv(qd, kd, vd, num_splits=ns, out=od, lse=ld, workspace=wsd)
        b0.record(stream)
        for _ in range(n_e):
            fa.fwd_splitkv(qd, kd, vd, num_splits=ns, out=od, lse=ld, workspace=wsd)
        b1.record(stream)
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        ms_d = b0.elapsed_time(b1) / n_e
        kv_bytes = 2.0 * wd.B * wd.H * wd.Nk * wd.d * 2
        extras[DECODE_EXTRA + "_splits"] = ns
        extras[DECODE_EXTRA + "_ms"] = ms_d
        extras[DECODE_EXTRA + "_kv_gbs"] = kv_bytes / (ms_d * 1e-3) / 1e9
        extras[DECODE_EXTRA + "_kv_frac_of_hbm"] = (kv_bytes / (ms_d * 1e-3) / 1e9
                                                    / load_peaks()[0].get("hbm_gbs", 6800.0))
        del qd, kd, vd, od, ld, wsd
        # grouped-query attention: the step's workload with 4 key/value heads
        hk = 4
        qg, dOg = (torch.randn((w.B, w.H, w.Nq, w.d), generator=g, device=dev,
                               dtype=torch.bfloat16) for _ in range(2))
        kg, vg = (torch.randn((w.B, hk, w.Nk, w.d), generator=g, device=dev,
                              dtype=torch.bfloat16) for _ in range(2))
        og = torch.empty_like(qg)
        lg = torch.empty(qg.shape[:3], dtype=torch.float32, device=dev)
        dqg, dkg, dvg = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)

        def gqa_step():
            fa.fwd(qg, kg, vg, out=og, lse=lg, **kw)
            fa.bwd(qg, kg, vg, og, lg, dOg, workspace=ws, dq=dqg, dk=dkg, dv=dvg, **kw)
        for _ in range(3):
            gqa_step()
        b0.record(stream)
        for _ in range(n_e):
            gqa_step()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        ms_g = b0.elapsed_time(b1) / n_e
        extras["gqa_b4h16kv4_n4096_d128_causal_fwdbwd_tflops"] = (f_fwd + f_bwd) / (ms_g * 1e-3) / 1e12
        del qg, dOg, kg, vg, og, lg, dqg, dkg, dvg
        # FP8 forward on the long-context workload: the e4m3 quantization and
        # the attention (e4m3 MMAs) timed apart; the attention against the
        # fp8 peak (2x the measured bf16 peak: the nominal fp8/bf16 ratio)
        qe, ke, ve = (torch.randn((we.B, we.H, we.Nq, we.d), generator=g, device=dev,
                                  dtype=torch.bfloat16) for _ in range(3))
        oe = torch.empty_like(qe)
        le = torch.empty(qe.shape[:3], dtype=torch.float32, device=dev)
        ws8 = torch.empty(fa.fa_fwd_fp8_workspace_size(we.B, we.H, we.H, we.Nq, we.Nk, we.d),
                          dtype=torch.uint8, device=dev)
        for _ in range(3):
            fa.fwd_fp8(qe, ke, ve, causal=True, out=oe, lse=le, workspace=ws8)
        ev8 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t_q, t_a = [], []
        for _ in range(n_e):
            ev8[0].record(stream)
            fa.fwd_fp8(qe, ke, ve, causal=True, out=oe, lse=le, workspace=ws8, stage=1)
            ev8[1].record(stream)
            fa.fwd_fp8(qe, ke, ve, causal=True, out=oe, lse=le, workspace=ws8, stage=2)
            ev8[2].record(stream)
            torch.cuda.synchronize(dev)
            t_q.append(ev8[0].elapsed_time(ev8[1]))
            t_a.append(ev8[1].elapsed_time(ev8[2]))
        fa.check_device_error(dev)
        f_e = flops(we)[0]
        fp8_peak = 2.0 * load_peaks()[0].get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        ms_a, ms_q = statistics.median(t_a), statistics.median(t_q)
        extras["fp8_" + we.name + "_fwd"] = {
            "attention_ms": ms_a, "quantize_ms": ms_q,
            "attention_tflops": f_e / (ms_a * 1e-3) / 1e12,
            "frac_of_fp8_peak": f_e / (ms_a * 1e-3) / 1e12 / fp8_peak,
            "with_quantize_tflops": f_e / ((ms_a + ms_q) * 1e-3) / 1e12,
            "fp8_peak_tflops": fp8_peak}
        del qe, ke, ve, oe, le, ws8
        # deterministic backward (query-outer dQ kernel, no reductions) on the
        # benchmark workload, timed per launch
        wsd = torch.empty(fa.fa_bwd_deterministic_workspace_size(w.B, w.H, w.Nq, w.d),
                          dtype=torch.uint8, device=dev)
        det_stages = ("preprocess", "dkdv", "dq")

        def det_bwd(ev=None):
            for i, st in enumerate(det_stages):
                if ev is not None:
                    ev[i].record(stream)
                fa.bwd(q, k, v, o, lse, dO, workspace=wsd, dq=dq, dk=dk, dv=dv,
                       deterministic=True, stage=st, **kw)
            if ev is not None:
                ev[3].record(stream)
        fa.fwd(q, k, v, out=o, lse=lse, **kw)
        for _ in range(3):
            det_bwd()
        evd = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_e)]
        for i in range(n_e):
            det_bwd(evd[i])
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        det_ms = {st: statistics.median(e[i].elapsed_time(e[i + 1]) for e in evd)
                  for i, st in enumerate(det_stages)}
        det_total = statistics.median(e[0].elapsed_time(e[3]) for e in evd)
        extras["deterministic_bwd_" + w.name] = {
            "ms": det_total, "stages_ms": det_ms,
            "tflops": f_bwd / (det_total * 1e-3) / 1e12,
            "flop_convention": "same 2.5x-forward count as fa_bwd (the kernels do 7/5 of it)"}
        del wsd
        # packed variable-length batch vs the same batch padded to its longest sequence
        lens = workloads.varlen_lengths(16, seed=2024)
        Hv, dv_ = 16, 128
        total, mx = sum(lens), max(lens)
        cu = torch.tensor([0] + list(__import__("itertools").accumulate(lens)), dtype=torch.int32,
                          device=dev)
        qv, kv_, vv, dOv = (torch.randn((Hv, total, dv_), generator=g, device=dev,
                                        dtype=torch.bfloat16) for _ in range(4))
        ov = torch.empty_like(qv)
        lv = torch.empty((Hv, total), dtype=torch.float32, device=dev)
        dqv, dkv, dvv = torch.empty_like(qv), torch.empty_like(kv_), torch.empty_like(vv)
        wsv = torch.empty(fa.fa_bwd_varlen_workspace_size(len(lens), Hv, total, mx, dv_),
                          dtype=torch.uint8, device=dev)

        def varlen_step():
            fa.fwd_varlen(qv, kv_, vv, cu, cu, causal=True, out=ov, lse=lv, max_seqlen_q=mx,
                          max_seqlen_k=mx)
            fa.bwd_varlen(qv, kv_, vv, ov, lv, dOv, cu, cu, causal=True, workspace=wsv, dq=dqv,
                          dk=dkv, dv=dvv, max_seqlen_q=mx, max_seqlen_k=mx)
        for _ in range(3):
            varlen_step()
        b0.record(stream)
        for _ in range(n_e):
            varlen_step()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        ms_v = b0.elapsed_time(b1) / n_e
        f_v = sum(3.5 * 4.0 * Hv * L * L * dv_ * 0.5 for L in lens)   # fwd + 2.5x bwd, causal
        del qv, kv_, vv, dOv, ov, lv, dqv, dkv, dvv, wsv
        # padded: B x max_len with the padding keys masked by the key bias
        B_ = len(lens)
        qp, kp, vp, dOp = (torch.randn((B_, Hv, mx, dv_), generator=g, device=dev,
                                       dtype=torch.bfloat16) for _ in range(4))
        bias_p = torch.zeros((B_, mx), dtype=torch.float32, device=dev)
        for i, L in enumerate(lens):
            bias_p[i, L:] = float("-inf")
        op = torch.empty_like(qp)
        lp = torch.empty(qp.shape[:3], dtype=torch.float32, device=dev)
        dqp, dkp, dvp = torch.empty_like(qp), torch.empty_like(kp), torch.empty_like(vp)
        wsp = torch.empty(fa.fa_bwd_workspace_size(B_, Hv, mx, mx, dv_), dtype=torch.uint8,
                          device=dev)

        def padded_step():
            fa.fwd(qp, kp, vp, key_bias=bias_p, causal=True, out=op, lse=lp)
            fa.bwd(qp, kp, vp, op, lp, dOp, key_bias=bias_p, causal=True, workspace=wsp, dq=dqp,
                   dk=dkp, dv=dvp)
        for _ in range(3):
            padded_step()
        b0.record(stream)
        for _ in range(n_e):
            padded_step()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        fa.check_device_error(dev)
        ms_p = b0.elapsed_time(b1) / n_e
        extras["varlen_16seq_h16_d128_causal"] = {
            "lengths": lens, "packed_ms": ms_v, "padded_ms": ms_p,
            "packed_effective_tflops": f_v / (ms_v * 1e-3) / 1e12,
            "padded_over_packed_time": ms_p / ms_v}
        del qp, kp, vp, dOp, bias_p, op, lp, dqp, dkp, dvp, wsp

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    med = {n: statistics.median(v) for n, v in parts.items()}
    bwd_main_tflops = f_bwd / (med["bwd_main"] * 1e-3) / 1e12
    fwd_tflops = f_fwd / (med["fwd"] * 1e-3) / 1e12
    # dominant kernel: the one with the largest share of the step
    dom = max(("fwd", "bwd_main"), key=lambda n: med[n])
    dom_flops = f_bwd if dom == "bwd_main" else f_fwd
    mean_dom = sum(parts[dom]) / len(parts[dom])
    achieved = dom_flops / (mean_dom * 1e-3) / 1e12
    # The timed region is milliseconds long and runs at the maximum SM clock
    # (see "clocks"), so the denominator is the burst peak; the sustained one
    # (a seconds-long loop under the power cap) is reported beside it.
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    traffic = TRAFFIC_BYTES.get(dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": "%s (burst bf16 dense)" % peak_src,
                "frac_of_sustained_peak": achieved / sustained,
                "frac_of_nominal_peak": achieved / NOMINAL_BF16_TFLOPS,
                "nominal_peak": NOMINAL_BF16_TFLOPS}
    cpu = cpu_baseline(w) if world == 1 else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16)",
        "config": bench_config(w, world),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "upload of step k+1, compute of step k and download of step k-1 "
                           "overlap (one copy stream per direction, two buffer sets)"},
        "gpu_launches": launches_per_step * args.steps,
        "parts_ms_median": med,
        "fwd_tflops": fwd_tflops,
        "bwd_main_tflops": bwd_main_tflops,
        "extras": extras,
        "clocks": clk.summary(),
        "peaks_source": peak_src,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# DRAM bytes per launch of the dominant kernels from an ncu capture, or None
# when the kernel changed since the counters were taken.
TRAFFIC_BYTES = {"fwd": 219976960 + 45267968, "bwd_main": 411727360 + 226045952}


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extra measurements (long-context forward, decode, GQA, ragged batch)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
