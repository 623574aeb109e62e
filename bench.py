"""Benchmark of the AWQ per-layer scale search on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step is the whole hot path over one seeded synthetic layer: channel
statistics, the alpha tables, the fused tcgen05 search over every alpha of
the grid, the reduction and argmin, and the final quantize + pack at the
kept scales, all through the C ABI.  The metric is layer-alpha-evals/s
(alphas searched per second); GFLOP/s and the tensor-core roofline fraction
of the search kernel are reported beside it.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; between steps a 512 MiB buffer is written to flush
the 126 MB L2 (outside the timed region).  With several GPUs (torchrun),
every rank searches its own layer (different seed): weak scaling, no
collective on the data path; the time is the max over ranks.

--impl reference times the CPU oracle (float64 numpy, the pages' algorithm
as written) on the same layer, each step the whole grid on the tiny and
notebook-shaped layers (a two-alpha sample on the larger ones).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synthetic import CONFIGS, config_by_name, make_layer  # noqa: E402

DEFAULT_CONFIG = "nb-4096x4096-n256"
METRIC = "AWQ search layer-alpha-evals/sec"

# The search kernel's DRAM bytes per launch (dram__bytes_read.sum +
# dram__bytes_write.sum) come from ncu captures summarised under profiles/,
# one "traffic-record:" line per capture, stamped with a hash of the kernel's
# sources.  A record counts only while those sources are unchanged; otherwise
# the line reports null.  Traffic far above W + X (each read once) would mean
# wasted re-reads.
SEARCH_SOURCES = ("post_weight_quantization_32_b300/csrc/awq_search.cu",
                  "post_weight_quantization_32_b300/csrc/awq_device.cuh")


def search_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in SEARCH_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def search_traffic(workload):
    """DRAM bytes of one search-kernel launch on `workload` from a profiles/
    record of the current kernel sources, else None."""
    import glob
    import re
    want = search_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                m = re.search(r"traffic-record: workload=(\S+) dram_bytes=(\d+) sources-sha256=([0-9a-f]+)",
                              line)
                if m and m.group(1) == workload and m.group(3) == want:
                    return int(m.group(2))
    return None


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1800.0), d.get("hbm_gbs", 6400.0), "measured"
    return 1800.0, 6400.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ.get("RANK", "0"))
        local = int(os.environ.get("LOCAL_RANK", "0"))
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, ws
    return None, 0, 1


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def world_max(v, dist, device):
    """The largest v over the ranks (v itself without a process group): the
    job takes as long as its slowest rank."""
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(n_alpha, world, ms):
    """Whole-job layer-alpha-evals/s: each rank searches its own layer over
    n_alpha alphas (weak scaling), all within the slowest rank's ms."""
    return n_alpha * world / (ms * 1e-3)


def run_ours(args, cfg, rank, world, dist):
    import post_weight_quantization_32_b300 as awq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    W, X = make_layer(cfg, seed=rank)
    Wd, Xd = W.to(dev), X.to(dev)
    out, n_in, N, na = cfg.out, cfg.in_, cfg.N, cfg.n_alpha
    ws = torch.empty(awq.awq_search_workspace_bytes(Wd.dtype, out, n_in, N, cfg.group, cfg.grid),
                     dtype=torch.uint8, device=dev)
    err = torch.empty(na, dtype=torch.float64, device=dev)
    best = torch.empty(1, dtype=torch.int32, device=dev)
    s_best = torch.empty(n_in, dtype=torch.float32, device=dev)
    nwords = (n_in * cfg.bits + 31) // 32
    qw = torch.empty((out, nwords), dtype=torch.int32, device=dev)
    sc = torch.empty((out, n_in // cfg.group), dtype=torch.float32, device=dev)
    zz = torch.empty((out, n_in // cfg.group), dtype=torch.uint8, device=dev)
    st = awq.new_status(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    ev_s0, ev_s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_s0.record(stream)   # torch creates the CUDA event at its first record
    ev_s1.record(stream)
    opts = awq.SearchOpts()
    opts.ev_search_start = ev_s0.cuda_event
    opts.ev_search_stop = ev_s1.cuda_event

    def step(W_, X_):
        # torch times only events it has recorded itself: record both here;
        # the library records them again around the search kernel
        ev_s0.record(stream)
        ev_s1.record(stream)
        awq.awq_search(W_, X_, cfg.bits, cfg.group, cfg.sym, cfg.grid, workspace=ws,
                       out_tensors=(err, best, s_best), dev_status=st, opts=opts, check=False)
        awq.awq_quantize_pack(W_, s_best, cfg.bits, cfg.group, cfg.sym, out_tensors=(qw, sc, zz),
                              dev_status=st, check=False)

    for _ in range(args.warmup):
        step(Wd, Xd)
    torch.cuda.synchronize()
    awq.check_status(st, "bench warm-up")
    if dist is not None:
        dist.barrier()
    step_ms, search_ms = [], []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        for _ in range(args.steps):
            flush.zero_()
            e0.record(stream)
            step(Wd, Xd)
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            search_ms.append(ev_s0.elapsed_time(ev_s1))
    torch.cuda.synchronize()
    awq.check_status(st, "bench")
    if dist is not None:
        dist.barrier()

    # end to end through the public API with host buffers: H2D of W and X from
    # pinned memory, the path, D2H of every result, every step
    Wh, Xh = W.pin_memory(), X.pin_memory()
    res_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (err, best, s_best, qw, sc, zz)]
    Wb, Xb = torch.empty_like(Wd), torch.empty_like(Xd)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0.record(stream)
        Wb.copy_(Wh, non_blocking=True)
        Xb.copy_(Xh, non_blocking=True)
        step(Wb, Xb)
        for h, d in zip(res_h, (err, best, s_best, qw, sc, zz)):
            h.copy_(d, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = W.numel() * W.element_size() + X.numel() * X.element_size()
    d2h = sum(t.numel() * t.element_size() for t in res_h)

    ms = world_max(sum(step_ms) / len(step_ms), dist, dev)
    e2e = world_max(sum(e2e_ms) / len(e2e_ms), dist, dev)
    t_search = world_max(sum(search_ms) / len(search_ms), dist, dev)
    return dict(ms=ms, e2e_ms=e2e, search_ms=t_search, h2d=h2d, d2h=d2h, clocks=clk.summary())


def run_oracle_sample(cfg, n_sample, seed=0):
    """Oracle wall time for n_sample alphas of the grid (spread over it; the
    whole grid when n_sample >= n_alpha), seconds, and the number of alphas.
    The oracle computes the statistics and the reference output X W^T once
    per call, as the pages' loop does, so a whole-grid call amortises them
    over every alpha and a sample does not."""
    from oracle import awq_oracle as O
    W, X = make_layer(cfg, seed=seed)
    Wn, Xn = W.float().numpy(), X.double().numpy()
    if n_sample >= cfg.n_alpha:
        idx = None
        n = cfg.n_alpha
    else:
        idx = set(np.linspace(0, cfg.n_alpha - 1, n_sample).round().astype(int).tolist())
        n = len(idx)
    t0 = time.perf_counter()
    O.awq_search(Wn, Xn, cfg.bits, cfg.group, cfg.grid, cfg.sym, alpha_index=idx)
    return time.perf_counter() - t0, n


def oracle_sample_size(cfg, requested):
    """Alphas in the oracle's timed sample: the requested count, else the
    whole grid where the oracle finishes it in seconds (the tiny and
    notebook-shaped layers), else two alphas."""
    if requested > 0:
        return requested
    return cfg.n_alpha if cfg.out * cfg.in_ * cfg.N <= 4096 * 4096 * 256 else 2


def oracle_sample_text(cfg, n):
    if n >= cfg.n_alpha:
        return ("the whole %d-alpha grid of the same layer in one oracle call (statistics and "
                "the reference output X W^T computed once, as the pages' loop does)" % cfg.n_alpha)
    return ("%d alphas of the %d-alpha grid of the same layer in one oracle call (statistics "
            "and the reference output X W^T computed once for the sample, so not amortised "
            "over the grid)" % (n, cfg.n_alpha))


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=[c.name for c in CONFIGS])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="alphas in the oracle's timed sample (0: the whole grid on the tiny and "
                         "notebook-shaped layers, two alphas on the larger ones)")
    ap.add_argument("--next-rows", action="store_true",
                    help="also time the clipping search, output power, wide-group searches, GPTQ "
                         "after AWQ and the checkpoint export on the same layer (one extra JSON "
                         "line each, rank 0)")
    args = ap.parse_args()
    cfg = config_by_name(args.config)
    dist, rank, world = _dist()
    tflops_peak, hbm_peak, peak_kind = _peaks()
    flops = cfg.search_flops
    conf = {"workload": cfg.name, "out": cfg.out, "in": cfg.in_, "N": cfg.N,
            "dtype_in": cfg.dtype, "bits": cfg.bits, "group": cfg.group,
            "quantizer": "sym" if cfg.sym else "asym", "n_alpha": cfg.n_alpha,
            "l2": "flushed between steps (512 MiB write)", "parallelism": "independent layers per rank"}

    if args.impl == "reference":
        if rank != 0:
            return
        n_s = oracle_sample_size(cfg, args.cpu_sample)
        times = []
        n = n_s
        for i in range(args.warmup + args.steps):
            t, n = run_oracle_sample(cfg, n_s)
            if i >= args.warmup:
                times.append(t)
        t = sum(times) / len(times)
        v = n / t
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "layer-alpha-evals/s",
                "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": conf,
                "cpu_baseline": {"value": v, "unit": "layer-alpha-evals/s", "cores": _cores(),
                                 "kind": "oracle", "sample": "each step: " + oracle_sample_text(cfg, n)},
                "e2e": {"value": v, "unit": "layer-alpha-evals/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    r = run_ours(args, cfg, rank, world, dist)
    if rank != 0:
        return
    n_alpha = cfg.n_alpha
    value = job_throughput(n_alpha, world, r["ms"])
    e2e_v = job_throughput(n_alpha, world, r["e2e_ms"])
    achieved = flops / (r["search_ms"] * 1e-3) / 1e12
    cpu_t, cpu_n = run_oracle_sample(cfg, oracle_sample_size(cfg, args.cpu_sample))
    # statistics, max|W| (with the s table and the X / s copies where the
    # search reads X pre-divided), the table of scalings, search, argmin,
    # pack; without the pre-divided mode a bf16 or fp32 X adds its fp16 copy
    xs_mode = (cfg.dtype in ("f16", "bf16") and cfg.N > 128 and cfg.group in (8, 16, 32, 64, 128)
               and cfg.n_alpha * cfg.N * cfg.in_ * 2 <= 64 * 2 ** 20)
    launches_per_step = 6 + (0 if xs_mode or cfg.dtype == "f16" else 1)
    line = {
        "metric": METRIC, "value": value, "unit": "layer-alpha-evals/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": conf,
        "gflops": flops / (r["ms"] * 1e-3) / 1e9,
        "search_kernel_ms": r["search_ms"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tflops_peak, "unit": "TFLOP/s",
                     "frac": achieved / tflops_peak, "traffic": search_traffic(cfg.name),
                     "kernel": "awq_search_kernel", "peak_kind": peak_kind + " (bf16 dense = fp16 dense)"},
        "cpu_baseline": {"value": cpu_n / cpu_t, "unit": "layer-alpha-evals/s", "cores": _cores(),
                         "kind": "oracle",
                         "sample": oracle_sample_text(cfg, cpu_n)},
        "e2e": {"value": e2e_v, "unit": "layer-alpha-evals/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": r["clocks"],
    }
    print(json.dumps(line))
    if args.next_rows:
        for extra in run_next_rows(args, cfg, tflops_peak, hbm_peak, peak_kind):
            print(json.dumps(extra))


# FP32 FMA lanes per SM and the maximum SM clock of a B300: the peak of the
# clipping search's quadratic forms, which run on the FMA pipe.
FP32_LANES_PER_SM, SM_MAX_GHZ = 128, 2.032


def run_next_rows(args, cfg, tflops_peak, hbm_peak, peak_kind):
    """Event-timed runs of the rows beyond the headline path, on the same
    layer and with the same L2 flush between runs."""
    import post_weight_quantization_32_b300 as awq

    dev = torch.device("cuda", 0)
    W, X = make_layer(cfg, seed=0)
    Wd, Xd = W.to(dev), X.to(dev)
    out, n_in, N, g = cfg.out, cfg.in_, cfg.N, cfg.group
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return sorted(ts)[len(ts) // 2]

    _, _, s_best = awq.awq_search(Wd, Xd, cfg.bits, g, cfg.sym, cfg.grid)
    steps_c = 10
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * SM_MAX_GHZ / 1e3          # TFLOP/s
    rows = []

    t = timed(lambda: awq.awq_clip_search(Wd, Xd, s_best, cfg.bits, g, cfg.sym, 20, steps_c,
                                          check=False))
    if cfg.dtype in ("f16", "bf16") and g == 128 and 32 <= N <= 256:
        # tensor cores: every factor's group errors times X / s, 2 N in out flops a factor
        fl = 2.0 * N * n_in * out * (steps_c + 1)
        clip_roof = {"bound": "tensor", "achieved": fl / t / 1e12, "peak": tflops_peak,
                     "unit": "TFLOP/s", "frac": fl / t / 1e12 / tflops_peak, "peak_kind": peak_kind}
    else:
        fl = 2.0 * out * n_in * g * (steps_c + 1) + 2.0 * n_in * g * N  # quadratic forms + Gram
        clip_roof = {"bound": "alu", "achieved": fl / t / 1e12, "peak": fp32_peak,
                     "unit": "TFLOP/s", "frac": fl / t / 1e12 / fp32_peak,
                     "peak_kind": "fp32 FMA lanes x max clock"}
    rows.append({"row": "clip_search", "metric": "group-factor-evals/s",
                 "value": out * (n_in // g) * (steps_c + 1) / t, "ms": t * 1e3,
                 "roofline": clip_roof})

    t = timed(lambda: awq.awq_output_power(Wd, Xd, check=False))
    fl = 2.0 * N * n_in * out
    rows.append({"row": "output_power", "metric": "layers/s", "value": 1.0 / t, "ms": t * 1e3,
                 "roofline": {"bound": "tensor", "achieved": fl / t / 1e12, "peak": tflops_peak,
                              "unit": "TFLOP/s", "frac": fl / t / 1e12 / tflops_peak,
                              "peak_kind": peak_kind}})

    for wide in (256, None):
        t = timed(lambda: awq.awq_search(Wd, Xd, cfg.bits, wide, cfg.sym, cfg.grid, check=False))
        fl = cfg.search_flops
        rows.append({"row": "search_group_%s" % ("row" if wide is None else wide),
                     "metric": "layer-alpha-evals/s", "value": cfg.n_alpha / t, "ms": t * 1e3,
                     "roofline": {"bound": "tensor", "achieved": fl / t / 1e12, "peak": tflops_peak,
                                  "unit": "TFLOP/s", "frac": fl / t / 1e12 / tflops_peak,
                                  "peak_kind": peak_kind + " (whole call incl. the range pass)"}})

    if g in (32, 64, 128):
        t = timed(lambda: awq.awq_gptq(Wd, Xd, s_best, cfg.bits, g, cfg.sym, check=False))
        # Hessian 2 N in^2, Cholesky in^3 / 3, triangular inverse in^3 / 3, error
        # propagation out in^2 (each in multiply-adds: 2 flops)
        fl = 2.0 * N * n_in ** 2 + 2.0 * n_in ** 3 / 3 * 2 + 2.0 * out * n_in ** 2 / 2 * 2
        rows.append({"row": "gptq_after_awq", "metric": "layers/s", "value": 1.0 / t,
                     "ms": t * 1e3,
                     "roofline": {"bound": "alu", "achieved": fl / t / 1e12, "peak": fp32_peak,
                                  "unit": "TFLOP/s", "frac": fl / t / 1e12 / fp32_peak,
                                  "peak_kind": "fp32 FMA lanes x max clock"}})

    qw, sc, z = awq.awq_quantize_pack(Wd, s_best, cfg.bits, g, cfg.sym)
    if 32 % cfg.bits == 0:
        t = timed(lambda: awq.awq_export_checkpoint(qw, sc, z, n_in, cfg.bits, g, check=False))
        # read: codes, fp32 steps, uint8 zeros; written: codes, fp16 steps, packed zeros
        nb = (qw.numel() * 4 + sc.numel() * 4 + z.numel()) + (qw.numel() * 4 + sc.numel() * 2
                                                              + z.numel() * cfg.bits // 8)
        rows.append({"row": "export_checkpoint", "metric": "GB/s", "value": nb / t / 1e9,
                     "ms": t * 1e3,
                     "roofline": {"bound": "hbm", "achieved": nb / t / 1e9, "peak": hbm_peak,
                                  "unit": "GB/s", "frac": nb / t / 1e9 / hbm_peak}})
    for r in rows:
        r.update({"workload": cfg.name, "steps": args.steps, "warmup": args.warmup,
                  "l2": "flushed between runs (512 MiB write)"})
    return rows


if __name__ == "__main__":
    main()
