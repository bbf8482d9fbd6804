"""Benchmark: exact attention forward, BF16, B=4, H=32, S=4096, D=128, causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one attn_fwd launch over the whole workload (inputs resident in
HBM). Prints ONE JSON line on rank 0 with the metric (TFLOP/s, FLOPs counted
as 4*B*Hq*Sq*Sk*D halved for causal), the roofline of the kernel against the
measured BF16 tensor peak, the end-to-end number through the public API with
host buffers (H2D of Q/K/V and D2H of O inside the timed region), the float64
CPU oracle timed on a bounded sample as a baseline, and the SM clocks sampled
during the timed region.

Multi-GPU (torchrun, one rank per GPU) runs independent replicas of the same
workload: attention forward shards with no exchange, so no data-path
collective exists; ranks only meet at barriers and a max over their times.
``--impl reference`` times the float64 oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_scaled_dot_flash_gb300 import synth  # noqa: E402

WORKLOAD = "bf16_causal_4k"
METRIC = "attention fwd TFLOP/s and % of GB300 BF16 peak (causal, S=4096, D=128)"
KERNEL_NAME = "attn_fwd_tc_kernel"
# key-range splits per workload (1 when absent): enough CTAs for 152 SMs
SPLITS = {"bf16_gqa_chunk_32k": 4}
# key-range splits of the serving workloads (1 when absent): with the decode
# kernels' longest-sequence-first order neither decode workload gains from splits
# (MLA decode: 218 us unsplit, 232 us with 2, 257 us with 4)
PAGED_SPLITS = {}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's ``value`` (a replicated job takes as long as
    its slowest rank); ``value`` itself outside a multi-rank process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_rank: float, max_seconds: float, world: int) -> float:
    """Whole-job throughput of ``world`` replicas that each do ``work_per_rank``."""
    return world * work_per_rank / max_seconds


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to ATTN_CLOCK_LOG_DIR (default: the system temp directory)
        log_dir = os.environ.get("ATTN_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"attn_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[3], f[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, val in zip(names[1:], r[3][1:]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


def make_device_tensor(a, kind, device):
    import torch
    t = torch.from_numpy(a.view("int16")).view(torch.bfloat16) if kind == "bf16" else torch.from_numpy(a)
    return t.to(device)


def make_device_inputs(w, device):
    import torch
    x = synth.make_inputs(w)

    def dev(a, kind):
        if a is None:
            return None
        if kind == "bf16":
            t = torch.from_numpy(a.view("int16")).view(torch.bfloat16)
        else:
            t = torch.from_numpy(a)
        return t.to(device)

    return x, {"q": dev(x["q"], w.dtype), "k": dev(x["k"], w.dtype), "v": dev(x["v"], w.dtype),
               "kv_lens": dev(x["kv_lens"], "i32"), "bias": dev(x["bias"], "f32")}


def read_traffic(w):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the kernel."""
    p = os.path.join(ROOT, "profiles", f"traffic_{w.name}.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        from exact_scaled_dot_flash_gb300 import build
        if d.get("kernel_source_sha") != build.kernel_source_digest(d.get("kernel_sources")):
            return None
        return d.get("dram_bytes_per_launch")
    except (OSError, ValueError, AttributeError):
        return None


def cpu_baseline(w, x, budget_s=12.0):
    """Float64 oracle on whole heads of the same workload, on all host cores."""
    import numpy as np
    import oracle
    wid = oracle.prepare(x["q"], x["k"], x["v"], kv_lens=x["kv_lens"], bias=x["bias"], dtype=w.dtype)
    per_head = w.flops() / (w.B * w.Hq)
    heads = [(b, h) for b in range(w.B) for h in range(w.Hq)]

    def run(hs):
        rows = np.array([(b, h, i) for b, h in hs for i in range(w.Sq)], dtype=np.int64)
        t0 = time.perf_counter()
        oracle.attention_rows(None, None, None, rows, mask=w.mask, scale=x["scale"], widened=wid)
        return time.perf_counter() - t0

    t1 = run(heads[:1])
    n = max(1, min(len(heads) - 1, int(budget_s / max(t1, 1e-3))))
    t = run(heads[1:1 + n])
    return {"value": n * per_head / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} whole (batch, head) slices of {w.name} ({w.Sq} query rows each, all "
                      f"{w.Sk} keys, causal), float64, {t:.1f} s on {os.cpu_count()} threads"}


def bench_reference(args):
    """Reference arm: the float64 oracle on the host cores, per-step bounded sample."""
    import numpy as np
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    wid = oracle.prepare(x["q"], x["k"], x["v"], kv_lens=x["kv_lens"], bias=x["bias"], dtype=w.dtype)
    threads = args.threads if args.threads > 0 else os.cpu_count()
    # per step: the last `nrows` query rows of every head of batch 0 in turn
    # (for causal workloads the last rows are the heaviest)
    rows_all = np.array([(0, h, i) for h in range(w.Hq) for i in range(w.Sq)], dtype=np.int64)
    L0 = min(max(int(x["kv_lens"][0]), 0), w.Sk) if x["kv_lens"] is not None else w.Sk

    def flops_of(rows):  # exact: 4 D FLOP per visible (query, key) pair
        vis = [min(L0, int(r[2]) + w.Sk - w.Sq + 1) if w.causal else L0 for r in rows]
        return float(sum(4.0 * max(n, 0) * w.D for n in vis))

    probe = rows_all[-64:]
    t0 = time.perf_counter()
    oracle.attention_rows(None, None, None, probe, mask=w.mask, scale=x["scale"], widened=wid, threads=threads)
    tp = max(time.perf_counter() - t0, 1e-4)
    budget = 90.0 / max(1, args.steps + args.warmup)
    nrows = int(max(16, min(len(rows_all), 64 * budget / tp)))
    rows = rows_all[-nrows:]
    for _ in range(args.warmup):
        oracle.attention_rows(None, None, None, rows, mask=w.mask, scale=x["scale"], widened=wid, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_rows(None, None, None, rows, mask=w.mask, scale=x["scale"], widened=wid, threads=threads)
    dt = time.perf_counter() - t0
    value = flops_of(rows) * args.steps / dt / 1e12
    sample = (f"the last {nrows} query rows of batch 0 of {w.name} per step (all their visible "
              f"keys), float64 oracle on {threads} threads")
    metric = METRIC if w.name == WORKLOAD else f"attention fwd TFLOP/s ({w.name})"
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
                       "D": w.D, "causal": w.causal},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def step_flops(w):
    """FLOPs of one step and their basis.

    Square causal problems use the nominal count 4*B*Hq*Sq*Sk*D / 2 of the
    headline metric. Otherwise (a causal window with Sq != Sk) the count is
    exact: 4*D per visible (query, key) pair, row i seeing min(Sk, i + Sk - Sq + 1)
    keys under the bottom-right causal mask.
    """
    if not w.causal or w.Sq == w.Sk:
        return w.flops(), "nominal 4*B*Hq*Sq*Sk*D" + (" / 2 (causal)" if w.causal else "")
    import numpy as np
    i = np.arange(w.Sq, dtype=np.int64)
    pairs = int(np.clip(i + (w.Sk - w.Sq) + 1, 0, w.Sk).sum())
    return 4.0 * w.B * w.Hq * w.D * pairs, "exact: 4*D per visible (query, key) pair"


def measure_f16_peak(device, n=8192, reps=10):
    """Dense F16 tensor throughput on this GPU: torch.matmul of two n x n f16
    matrices (2 n^3 FLOP), best of ``reps`` timed with CUDA events. Serves as
    the roofline denominator of F16 workloads (the BF16 one is the driver's
    measurement in MEASURED_PEAKS.json)."""
    import torch
    a = torch.randn(n, n, device=device, dtype=torch.float16)
    b = torch.randn(n, n, device=device, dtype=torch.float16)
    c = torch.empty(n, n, device=device, dtype=torch.float16)
    for _ in range(3):
        torch.matmul(a, b, out=c)
    best = float("inf")
    for _ in range(reps):
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record()
        torch.matmul(a, b, out=c)
        e_ev.record()
        torch.cuda.synchronize()
        best = min(best, s_ev.elapsed_time(e_ev))
    del a, b, c
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def padding_ideal(w, x, peak_tflops, hbm_gbs):
    """Exact work of a key-padding workload: 4*D FLOP per visible (query, key)
    pair, and the bytes needed once (Q, O, the valid K/V rows, the bias once,
    kv_lens); the ideal time is the larger of FLOP/peak and bytes/bandwidth."""
    import numpy as np
    es = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
    L = np.clip(np.asarray(x["kv_lens"], dtype=np.int64), 0, w.Sk)
    if w.causal:
        i = np.arange(w.Sq, dtype=np.int64)
        vis = np.minimum(L[:, None], np.clip(i[None, :] + (w.Sk - w.Sq) + 1, 0, w.Sk)).sum()
    else:
        vis = int(L.sum()) * w.Sq
    flops = 4.0 * w.D * w.Hq * float(vis)
    nbytes = 2 * w.B * w.Hq * w.Sq * w.D * es + 2 * int(L.sum()) * w.Hkv * w.D * es + 4 * w.B
    if w.bias:
        nbytes += w.bias_b * w.bias_h * w.Sq * w.Sk * 4
    t_flop = flops / (peak_tflops * 1e12)
    t_mem = nbytes / (hbm_gbs * 1e9)
    return {"exact_flops": flops, "algorithmic_bytes": nbytes, "ideal_us": max(t_flop, t_mem) * 1e6,
            "bound_of_ideal": "tensor" if t_flop >= t_mem else "hbm"}


def bench_gpu(args):
    import torch
    from exact_scaled_dot_flash_gb300 import attn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    w = synth.WORKLOADS[args.workload]
    x, t = make_device_inputs(w, device)
    q, k, v, lens, bias = t["q"], t["k"], t["v"], t["kv_lens"], t["bias"]
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)
    scale = x["scale"]
    causal = w.causal

    splits = args.splits if args.splits else SPLITS.get(w.name, 1)
    ws = None
    if splits > 1:
        shp = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, 1, 1)
        ws = torch.empty(attn.split_workspace_bytes(shp, splits), dtype=torch.uint8, device=device)

    def step():
        # the current stream: the bench's own, or the capture stream of a CUDA graph
        attn.fwd(q, k, v, causal=causal, kv_lens=lens, bias=bias, scale=scale, out=out,
                 stream=torch.cuda.current_stream(device), num_splits=splits, workspace=ws)

    bwd_bufs = None
    if args.pass_ == "bwd":
        # inputs of the backward: the forward's output and LSE, and a seeded dL/dO
        g = make_device_tensor(synth.to_storage(synth.normal_f32(w.seed, 7, (w.B, w.Hq, w.Sq, w.D)), w.dtype),
                               w.dtype, device)
        fo, flse = attn.fwd(q, k, v, causal=causal, kv_lens=lens, bias=bias, scale=scale, return_lse=True)
        bshp = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, *(x["bias"].shape[:2] if w.bias else (1, 1)))
        bws = torch.empty(max(1, attn.bwd_workspace_bytes(bshp)), dtype=torch.uint8, device=device)
        bwd_bufs = dict(out=fo, dout=g, lse=flse, dq=torch.empty_like(q), dk=torch.empty_like(k),
                        dv=torch.empty_like(v))

        def step():  # noqa: F811 - the timed step is the backward
            attn.bwd(q, k, v, bwd_bufs["out"], bwd_bufs["dout"], bwd_bufs["lse"], causal=causal, kv_lens=lens,
                     bias=bias, scale=scale, workspace=bws, stream=stream, dq=bwd_bufs["dq"],
                     dk=bwd_bufs["dk"], dv=bwd_bufs["dv"])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    attn.device_status(device.index, clear=True)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = None
    if args.graph:  # the K steps captured once, replayed as one graph launch
        if args.pass_ != "fwd" or args.l2_flush:
            raise SystemExit("--graph times the forward without --l2-flush")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                step()
        torch.cuda.synchronize()
        graph.replay()  # one untimed replay
        torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device) if args.l2_flush else None
    per_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if args.l2_flush else None
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_id = vis.split(",")[device.index] if vis else str(device.index)
    with ClockSampler(smi_id) as clocks:
        barrier()
        torch.cuda.synchronize()
        if per_step:  # each step timed alone, 256 MiB written between steps to evict L2
            for s_ev, e_ev in per_step:
                flush.zero_()
                s_ev.record(stream)
                step()
                e_ev.record(stream)
        else:
            start.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for _ in range(args.steps):
                    step()
            end.record(stream)
        torch.cuda.synchronize()
        barrier()
    elapsed_ms = (sum(s_ev.elapsed_time(e_ev) for s_ev, e_ev in per_step) if per_step
                  else start.elapsed_time(end))
    status = attn.device_status(device.index, clear=True)
    if status:
        raise RuntimeError(f"kernel status flags {status:#x} during the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, device)
    ms = elapsed_ms / args.steps
    flops, flops_basis = step_flops(w)
    if args.pass_ == "bwd":  # nominal backward work: 2.5x the forward's (5 matmuls for 2)
        flops, flops_basis = 2.5 * flops, "2.5 x forward (" + flops_basis + ")"
    value = replica_throughput(flops, ms * 1e-3, world) / 1e12

    # end to end through the public API with host buffers (pinned), copies inside
    e2e = None
    if not args.no_e2e and args.pass_ == "fwd":
        hosts = [None if a is None else a.cpu().pin_memory() for a in (q, k, v, lens, bias)]
        qh, kh, vh, lh, bh = hosts
        oh = torch.empty(qh.shape, dtype=qh.dtype, pin_memory=True)
        e2e_steps = max(3, min(10, args.steps))

        def e2e_step():
            if splits == 1:
                attn.fwd(qh, kh, vh, causal=causal, kv_lens=lh, bias=bh, scale=scale, out=oh)
            else:  # the same public call on device copies made inside the step
                up = [None if a is None else a.to(device, non_blocking=True) for a in (qh, kh, vh, lh, bh)]
                o = attn.fwd(up[0], up[1], up[2], causal=causal, kv_lens=up[3], bias=up[4], scale=scale,
                             num_splits=splits, workspace=ws)
                oh.copy_(o, non_blocking=True)
                torch.cuda.current_stream(device).synchronize()

        for _ in range(5):  # untimed: first-use costs of the pinned buffers and streams
            e2e_step()
        # three timed windows of e2e_steps steps; the median window is reported
        # (a host-side disturbance in one window does not decide the number)
        windows = []
        for _ in range(3):
            barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(e2e_steps):
                e2e_step()
            torch.cuda.synchronize()
            windows.append((time.perf_counter() - t0) / e2e_steps)
        e2e_s = max_over_ranks(statistics.median(windows), device)
        h2d = sum(a.numel() * a.element_size() for a in hosts if a is not None)
        d2h = oh.numel() * oh.element_size()
        e2e = {"value": replica_throughput(flops, e2e_s, world) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
               "windows_ms": [round(wnd * 1e3, 4) for wnd in windows], "timing": f"median of 3 windows of {e2e_steps} steps",
               "path": ("attn.fwd on pinned host tensors -> attn_fwd_host: chunked H2D copies, attn_fwd per "
                        "chunk and D2H copies overlapped on three streams, sync") if splits == 1 else
                       "attn.fwd_split on device copies made inside the step: H2D, attn_fwd_split, D2H, sync"}

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_desc = f"{peak_kind} bf16 dense burst"
    if w.dtype == "f16":  # F16 runs against an F16 peak measured in this run
        peak = measure_f16_peak(device)
        peak_desc = "f16 dense burst measured in this run (torch.matmul f16 8192^3, best of 10)"
    achieved = flops / (ms * 1e-3) / 1e12
    traffic = read_traffic(w)
    hbm_gbs = w.io_bytes() / (ms * 1e-3) / 1e9
    line = {
        "metric": (METRIC if w.name == WORKLOAD and args.pass_ == "fwd"
                   else f"attention {args.pass_} TFLOP/s ({w.name})"), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "causal": w.causal, "key_padding": bool(w.mask & synth.MASK_KEY_PADDING),
                   "bias": [w.bias_b, w.bias_h] if w.bias else None, "parallelism": f"replicas x{world}",
                   "num_splits": splits, "flops_basis": flops_basis,
                   "l2": ("L2 flushed: 256 MiB written between timed steps, each step timed alone"
                          if args.l2_flush else
                          f"inputs larger than L2: {w.io_bytes() / 2**20:.0f} MiB per step vs 129 MB L2, no flush"
                          if w.io_bytes() > 129e6 else
                          f"working set {w.io_bytes() / 2**20:.1f} MiB fits in L2 (L2-hot steps)"),
                   "launch": "CUDA graph of the K steps, one replay" if graph is not None else "eager"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": peak_desc,
                     "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                     "kernel": KERNEL_NAME if w.dtype != "f32" else "attn_fwd_f32_kernel",
                     "hbm_gbs_algorithmic": hbm_gbs,
                     "hbm_frac": hbm_gbs / float(peaks["hbm_gbs"])},
        "e2e": e2e,
        "gpu_launches": args.steps * (3 if args.pass_ == "bwd" else (2 if splits > 1 else 1)),
        "clocks": clocks.summary(),
    }
    if w.mask & synth.MASK_KEY_PADDING and args.pass_ == "fwd":
        ideal = padding_ideal(w, x, peak, float(peaks["hbm_gbs"]))
        ideal["frac_of_ideal"] = ideal["ideal_us"] / (ms * 1e3)
        line["roofline"]["padding"] = ideal
    if args.pass_ == "bwd" and w.dtype != "f32" and w.D in (64, 128):
        line["roofline"].update({"kernel": "dkdv_tc_kernel + dq_tc_kernel", "traffic": None})
    elif args.pass_ == "bwd":
        # the fp32 FMA backward: its roofline is the FMA pipes' peak,
        # 152 SMs x 128 lanes x 2 FLOP x the SM clock seen under load
        mhz = (line["clocks"] or {}).get("sm_mhz") or 2070.0
        alu_peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
        line["roofline"].update({"bound": "alu", "peak": alu_peak, "frac": achieved / alu_peak,
                                 "peak_kind": f"fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz",
                                 "frac_of_sustained": None, "kernel": "dkdv_kernel + dq_kernel",
                                 "traffic": None})
    if world == 1 and not args.no_cpu_baseline and w.name == WORKLOAD and args.pass_ == "fwd":
        line["cpu_baseline"] = cpu_baseline(w, x)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_paged(args):
    """Paged-cache attention (attn_paged_fwd) on a serving-shaped workload: one
    step = one call over the packed queries of every sequence."""
    import numpy as np
    import torch
    from exact_scaled_dot_flash_gb300 import attn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    is_mla = args.workload in synth.MLA_WORKLOADS
    w = synth.MLA_WORKLOADS[args.workload] if is_mla else synth.PAGED_WORKLOADS[args.workload]
    x = synth.make_mla_inputs(w) if is_mla else synth.make_paged_inputs(w)
    names = ("q", "qp", "latent", "kpos") if is_mla else ("q", "k_cache", "v_cache")
    t = [make_device_tensor(x[n], w.dtype, device) for n in names]
    ints = {n: torch.from_numpy(x[n]).to(device) for n in ("block_table", "seq_lens", "q_offsets")}
    pos = torch.from_numpy(x["positions"]).to(device) if x["positions"] is not None else None
    nq_s = np.diff(x["q_offsets"])
    max_q = int(nq_s.max()) if len(nq_s) else 0
    out = torch.empty_like(t[0])
    stream = torch.cuda.current_stream(device)
    splits = args.splits if args.splits else PAGED_SPLITS.get(w.name, 1)
    if is_mla:
        shp = attn.MlaShape(w.num_seqs, int(x["q_offsets"][-1]), w.H, w.R, w.Pd, w.page_size,
                            int(x["latent"].shape[0]), int(x["block_table"].shape[1]), max_q)
        need = attn.mla_workspace_bytes(shp, splits)
    else:
        shp = attn.PagedShape(w.num_seqs, int(x["q_offsets"][-1]), w.Hq, w.Hkv, w.D, w.page_size,
                              int(x["k_cache"].shape[0]), int(x["block_table"].shape[1]), max_q)
        need = attn.paged_workspace_bytes(shp, splits)
    pws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    # the paths the library takes for this call (see attn_paged_fwd / attn_paged_mla)
    decode = (not is_mla) and max_q * (w.Hq // w.Hkv) <= 8
    if is_mla:
        tensor = (w.dtype != "f32" and w.R in (256, 512) and w.Pd in (0, 64) and w.page_size % 8 == 0
                  and (64 % w.page_size == 0 or w.page_size % 64 == 0))
        # the backward's tensor-core kernels gather 128-key blocks
        tensor_bwd = (w.dtype != "f32" and w.R in (256, 512) and w.Pd in (0, 64) and w.page_size % 8 == 0
                      and (128 % w.page_size == 0 or w.page_size % 128 == 0))
    else:
        tensor = (w.dtype != "f32" and w.D in (64, 128) and w.page_size % 8 == 0
                  and (128 % w.page_size == 0 or w.page_size % 128 == 0))
    launches = 2 if need > 0 and (decode or (is_mla and tensor)) else 1
    bwd = args.pass_ == "bwd"
    if bwd:  # the forward's output and statistics once, untimed; a random dL/dO
        call = attn.paged_mla if is_mla else attn.paged_fwd
        fo, flse = call(*t, ints["block_table"], ints["seq_lens"], ints["q_offsets"], positions=pos,
                        causal=w.causal, scale=x["scale"], max_queries=max_q, return_lse=True)
        g = make_device_tensor(synth.to_storage(synth.normal_f32(w.seed, 9, x["q"].shape), w.dtype), w.dtype, device)
        need = attn.mla_bwd_workspace_bytes(shp) if is_mla else attn.paged_bwd_workspace_bytes(shp)
        pws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        # preprocess, page-index count / scan / fill / sort, key-major and query-major kernels
        # (tensor-core paths add the FMA key-major pass over shared pages)
        launches = 8 if (tensor_bwd if is_mla else tensor) else 7

    def step():
        if bwd:
            call = attn.paged_mla_bwd if is_mla else attn.paged_bwd
            call(*t, ints["block_table"], ints["seq_lens"], ints["q_offsets"], g, out=fo, lse=flse, positions=pos,
                 causal=w.causal, scale=x["scale"], max_queries=max_q, workspace=pws, stream=stream)
            return
        call = attn.paged_mla if is_mla else attn.paged_fwd
        call(*t, ints["block_table"], ints["seq_lens"], ints["q_offsets"], positions=pos, causal=w.causal,
             scale=x["scale"], max_queries=max_q, out=out, stream=stream, num_splits=splits, workspace=pws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    attn.device_status(device.index, clear=True)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_id = vis.split(",")[device.index] if vis else str(device.index)
    with ClockSampler(smi_id) as clocks:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    elapsed_ms = start.elapsed_time(end)
    if attn.device_status(device.index, clear=True):
        raise RuntimeError("kernel status flags set during the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, device)
    ms = elapsed_ms / args.steps
    # exact work: 4*D FLOP per visible (query, key) pair and query head
    pairs = 0
    for s_, L in enumerate(x["seq_lens"]):
        n = int(nq_s[s_])
        pq = (x["positions"][x["q_offsets"][s_]:x["q_offsets"][s_ + 1]] if x["positions"] is not None
              else np.arange(L - n, L))
        pairs += int(np.minimum(L, np.asarray(pq, dtype=np.int64) + 1).clip(min=0).sum()) if w.causal else n * int(L)
    es = {"f32": 4, "f16": 2, "bf16": 2}[w.dtype]
    nqt, nkt = int(x["q_offsets"][-1]), int(x["seq_lens"].sum())
    if is_mla:  # 2(R + Pd) for the score, 2R for the latent sum, per pair and head
        flops = (2.0 * (w.R + w.Pd) + 2.0 * w.R) * w.H * pairs
        nbytes = (nkt * (w.R + w.Pd) + nqt * w.H * (2 * w.R + w.Pd)) * es
    else:
        flops = 4.0 * w.D * w.Hq * pairs
        nbytes = (2 * nkt * w.Hkv * w.D + 2 * nqt * w.Hq * w.D) * es
    flops_basis = "exact: per visible (query, key) pair and head"
    if bwd:  # nominal backward work: 2.5x the forward's (5 matmuls for 2)
        flops, flops_basis = 2.5 * flops, "2.5 x forward (" + flops_basis + ")"
        nbytes *= 2  # inputs and out/dout read, gradients written: twice the forward's bytes
    value = replica_throughput(flops, ms * 1e-3, world) / 1e12
    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    mhz = (clocks.summary() or {}).get("sm_mhz") or 2070.0
    alu_peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
    tf = flops / (ms * 1e-3) / 1e12
    # roofline of the path taken: decode-shaped paged calls (<= 8 rows per
    # sequence and kv head) stream the cache (HBM); prefill-shaped F16/BF16
    # paged calls with D in {64, 128} run on the tensor cores; tensor-core MLA
    # is held to whichever of the tensor and HBM rooflines binds (the larger
    # ideal time); the rest runs on the fp32 FMA pipes
    mla_hbm = is_mla and tensor and nbytes / float(peaks["hbm_gbs"]) > flops / (float(peaks["bf16_tflops"]) * 1e3)
    # the paged backward: tensor cores for F16/BF16 paged attention with D in
    # {64, 128} (HBM-bound when decode-shaped), the fp32 FMA kernels otherwise;
    # the MLA backward on the tensor cores is held to whichever of the tensor
    # and HBM rooflines binds (the larger ideal time)
    bwd_tc = bwd and not is_mla and tensor
    mla_bwd_tc = bwd and is_mla and tensor_bwd
    tc_names = (("paged_dkdv_narrow_kernel or paged_dkdv_stream_kernel" if decode else "paged_dkdv_tc_kernel")
                + " + paged_dq_tc_kernel (+ FMA pass over shared pages), whole call")
    if mla_bwd_tc:
        pk, bw = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
        names = "mla_bwd_tc_kernel key-major + query-major (+ FMA pass over shared pages), whole call"
        if nbytes / bw > flops / (pk * 1e3):
            roof = {"bound": "hbm", "achieved": gbs, "peak": bw, "unit": "GB/s", "frac": gbs / bw,
                    "peak_kind": f"{peak_kind} HBM copy", "kernel": names}
        else:
            roof = {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                    "peak_kind": f"{peak_kind} bf16 dense burst", "kernel": names}
    elif bwd and bwd_tc and decode:
        roof = {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": gbs / float(peaks["hbm_gbs"]), "peak_kind": f"{peak_kind} HBM copy", "kernel": tc_names}
    elif bwd_tc:
        pk = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                "peak_kind": f"{peak_kind} bf16 dense burst", "kernel": tc_names}
    elif bwd:
        roof = {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                "peak_kind": f"fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz",
                "kernel": "dkdv_kernel + dq_kernel (paged backward, whole call)"}
    elif decode or mla_hbm:
        roof = {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": gbs / float(peaks["hbm_gbs"]), "peak_kind": f"{peak_kind} HBM copy",
                "kernel": "mla_tc_kernel" if is_mla else ("paged_tc_kernel" if tensor else "paged_decode_kernel")}
    elif tensor:
        pk = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                "peak_kind": f"{peak_kind} bf16 dense burst",
                "kernel": "mla_tc_kernel" if is_mla else "paged_tc_kernel"}
    else:
        roof = {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                "peak_kind": f"fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz",
                "kernel": "mla_fwd_kernel" if is_mla else "paged_fwd_kernel"}
    roof.update({"traffic": None, "algorithmic_bytes": nbytes})
    heads = {"H": w.H, "R": w.R, "Pd": w.Pd} if is_mla else {"Hq": w.Hq, "Hkv": w.Hkv, "D": w.D}
    line = {
        "metric": f"{'MLA' if is_mla else 'paged attention'}{' bwd' if bwd else ''} TFLOP/s ({w.name})",
        "value": value, "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, **heads, "page_size": w.page_size, "ctx_range": list(w.ctx_range), "q_range": list(w.q_range),
                   "queries": int(x["q_offsets"][-1]), "keys": int(x["seq_lens"].sum()),
                   "parallelism": f"replicas x{world}", "flops_basis": flops_basis,
                   "num_splits": splits if (decode or (is_mla and tensor)) and not bwd else 1,
                   "l2": f"cache read {nbytes / 2**20:.0f} MiB per step"},
        "roofline": roof, "hbm_gbs_algorithmic": gbs, "e2e": None,
        "gpu_launches": args.steps * launches, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=sorted(synth.WORKLOADS) + sorted(synth.PAGED_WORKLOADS) + sorted(synth.MLA_WORKLOADS))
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"],
                    help="time the forward (default) or the backward (attn_bwd, attn_paged_bwd, "
                         "attn_paged_mla_bwd) of the workload")
    ap.add_argument("--splits", type=int, default=0,
                    help="key-range splits (attn_fwd_split); 0 = the workload's default")
    ap.add_argument("--threads", type=int, default=0,
                    help="host threads of the reference arm's oracle (0 = all cores)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the K forward steps in a CUDA graph and time one replay")
    ap.add_argument("--l2-flush", action="store_true",
                    help="write 256 MiB between steps and time each step alone (L2-cold inputs)")
    args = ap.parse_args()
    paged = args.workload in synth.PAGED_WORKLOADS or args.workload in synth.MLA_WORKLOADS
    if args.impl == "reference" and paged:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the dense workloads"}))
    elif args.impl == "reference":
        bench_reference(args)
    elif paged:
        bench_paged(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
