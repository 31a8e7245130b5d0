"""Benchmark: exact attention forward + backward on one GB300, B=1 H=32 N=8192 d=128 causal.

One step = one pass of the whole hot path on one batch of synthetic bf16
input already resident in HBM: fattn_fwd (O, LSE) then fattn_bwd (D
preprocess, dK/dV/dQ main kernel, dQ convert).  FLOPs follow the workload's
convention: forward 4*B*H*N^2*d, backward 2.5x that, both halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own copy of the workload on its
own GPU (independent problems, no collective on the data path: weak scaling);
the timed region is bracketed by a barrier and a synchronize on both sides and
the slowest rank's time is used.

--impl reference times the fp64 CPU oracle, as it stands, on the host cores
(one step = forward + backward of a bounded sample of the workload: one head,
the first PREFIX tokens of the causal sequence).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from online_softmax_08_gb300.inputs import (DECODE_WORKLOADS, HEADLINE,  # noqa: E402
                                            HOST_WORKLOADS, SOFTMAX_WORKLOADS, VARLEN_WORKLOADS,
                                            WORKLOADS, default_scale, make_host_inputs,
                                            make_inputs, make_softmax_input, make_varlen_inputs,
                                            varlen_lengths)

METRIC = "attention fwd/bwd TFLOP/s, N=8192 d=128 bf16 causal; % of GB300 BF16 peak"
UNIT = "TFLOP/s"
REF_PREFIX = 2048        # tokens of one head per reference-arm step
CPU_BASELINE_SECONDS = 12.0


def flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d * (0.5 if causal else 1.0)
    return f, 2.5 * f


def job_tflops(world, step_flops, ms_per_step):
    """Whole-job throughput: every rank runs one full workload per step, and
    ms_per_step is the slowest rank's."""
    return world * step_flops / (ms_per_step * 1e-3) / 1e12


def measured_traffic(kernel):
    """DRAM bytes per launch of ``kernel`` from the committed ncu capture, or None
    when the kernel's sources changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic_b1h32_n8192_d128_causal.json")
    try:
        with open(path) as f:
            entry = json.load(f)["kernels"][kernel]
        m = hashlib.sha256()
        for name in entry["sources"]:
            with open(os.path.join(ROOT, "online_softmax_08_gb300", "csrc", name), "rb") as f:
                m.update(f.read())
        return entry["bytes"] if m.hexdigest() == entry["sha256"] else None
    except Exception:
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


def _clean(x):
    """JSON-safe copy: NaN and inf become null."""
    if isinstance(x, dict):
        return {k: _clean(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [_clean(v) for v in x]
    if isinstance(x, float) and not math.isfinite(x):
        return None
    return x


# ------------------------------------------------------------------ multi-rank plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """Largest value of a float over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running.  Each
    sample carries nvidia-smi's timestamp; the figures are taken from the samples
    that fall inside the timed region (region_start .. region_end), or from all
    samples when the region is shorter than the sampling interval."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def region_start(self):
        import datetime
        self.t_start = datetime.datetime.now()

    def region_end(self):
        import datetime
        self.t_end = datetime.datetime.now()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []  # (time or None, sm MHz, max MHz, active reasons)
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm, smax = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            try:
                when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                when = None
            active = {name for name, val in zip(names, parts[6:10]) if val.lower().startswith("active")}
            samples.append((when, sm, smax, active))
        inside = [x for x in samples
                  if x[0] is not None and self.t_start is not None and self.t_end is not None
                  and self.t_start <= x[0] <= self.t_end]
        use = inside or samples
        reasons = set().union(*(x[3] for x in use)) if use else set()
        return {"sm_mhz": statistics.median(x[1] for x in use) if use else None,
                "sm_max_mhz": max(x[2] for x in use) if use else None,
                "reasons": sorted(reasons), "samples": len(samples),
                "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ reference arm / CPU baseline

def oracle_step(q, k, v, do, scale, causal, prefix):
    """fp64 oracle forward + backward on one head, the first ``prefix`` tokens."""
    import oracle
    sl = (slice(0, 1), slice(0, 1), slice(0, prefix))
    f64 = lambda t: t[sl].to(torch.float64).numpy()
    qh, kh, vh, doh = f64(q), f64(k), f64(v), f64(do)
    oracle.attention_fwd(qh, kh, vh, scale, causal)
    oracle.attention_bwd(qh, kh, vh, doh, scale, causal)
    f, b = flops(1, 1, prefix, q.shape[-1], causal)
    return f + b


def cpu_baseline(inputs, scale, causal, min_seconds=CPU_BASELINE_SECONDS, prefix=REF_PREFIX):
    import oracle
    q, k, v, do = inputs
    done, t0 = 0.0, time.perf_counter()
    steps = 0
    while True:
        done += oracle_step(q, k, v, do, scale, causal, prefix)
        steps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": done / el / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": "fp64 oracle forward+backward of head 0, first %d tokens of the causal "
                      "sequence, repeated %d times (%.1f s)" % (prefix, steps, el)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOADS[HEADLINE]
    d = w["d"]
    q, k, v, do = make_inputs(1, 1, REF_PREFIX, d, w["seed"], w["q_std"], w["v_dist"], with_do=True)
    scale = default_scale(d)
    for _ in range(args.warmup):
        oracle_step(q, k, v, do, scale, True, REF_PREFIX)
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        total += oracle_step(q, k, v, do, scale, True, REF_PREFIX)
    el = time.perf_counter() - t0
    import oracle
    value = total / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "B": 1, "H": 1, "N": REF_PREFIX, "d": d, "causal": True,
                   "sample": "one head, first %d tokens" % REF_PREFIX},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": "fp64 oracle forward+backward, one head, first %d tokens of "
                                   "the causal sequence per step" % REF_PREFIX},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    from online_softmax_08_gb300 import fattn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    fattn.load()

    w = WORKLOADS[args.workload]
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"][-1]
    if args.causal != "default":  # profiling: another masking mode the workload lists
        causal = args.causal == "yes"
        if causal not in w["causal"]:
            raise SystemExit("workload %s has no %s mode" % (args.workload, args.causal))
    scale = default_scale(d)
    f_fwd, f_bwd = flops(B, H, N, d, causal)
    do_fwd, do_bwd = args.passes in ("both", "fwd"), args.passes in ("both", "bwd")
    host = make_inputs(B, H, N, d, w["seed"] + 1000 * rank, w["q_std"], w["v_dist"], with_do=True)
    q, k, v, do = (x.to(device) for x in host)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fattn.fattn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    K = args.steps
    fwd_ev = [(ev(), ev()) for _ in range(K)]
    bwd_ev = [[ev() for _ in range(4)] for _ in range(K)]

    if not do_fwd:  # the backward alone still needs a forward's O and LSE
        fattn.fattn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)

    def step(i=None):
        if do_fwd:
            if i is not None:
                fwd_ev[i][0].record(stream)
            fattn.fattn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)
            if i is not None:
                fwd_ev[i][1].record(stream)
        if do_bwd:
            if i is not None:
                fattn.fattn_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, ws,
                                   ws_bytes, bwd_ev[i], stream)
            else:
                fattn.fattn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, ws,
                                ws_bytes, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    for pair in fwd_ev:  # materialise event handles outside the timed region
        pair[0].record(stream)
        pair[1].record(stream)
    for evs in bwd_ev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(device)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    t0, t1 = ev(), ev()
    clocks.region_start()
    t0.record(stream)
    for i in range(K):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks.region_end()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, device)
    assert fattn.fattn_device_error() == 0, "an in-kernel wait timed out"

    nan = float("nan")
    # per-kernel times over the K timed steps: the median is the figure used
    # (steadier against one slow launch), the mean is reported beside it
    fwd_t = [a.elapsed_time(b) for a, b in fwd_ev] if do_fwd else [nan]
    pre_t = [e[0].elapsed_time(e[1]) for e in bwd_ev] if do_bwd else [nan]
    main_t = [e[1].elapsed_time(e[2]) for e in bwd_ev] if do_bwd else [nan]
    conv_t = [e[2].elapsed_time(e[3]) for e in bwd_ev] if do_bwd else [nan]
    fwd_ms, pre_ms, main_ms, conv_ms = (statistics.median(t) for t in (fwd_t, pre_t, main_t, conv_t))
    means = {name: statistics.mean(t) for name, t in
             (("fwd_ms", fwd_t), ("preprocess_ms", pre_t), ("main_ms", main_t),
              ("convert_ms", conv_t))}
    ms_per_step = elapsed_ms / K
    step_flops = (f_fwd if do_fwd else 0.0) + (f_bwd if do_bwd else 0.0)
    value = job_tflops(world, step_flops, ms_per_step)
    peak_tf, peak_hbm, peak_src = peaks()

    # the dominant kernel by time is the backward main kernel; its algorithmic
    # work is the 2.5x-forward FLOP count of the workload
    main_tf = f_bwd / (main_ms * 1e-3) / 1e12
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    rows = B * H * N
    fwd_bytes = 4 * rows * d * 2 + rows * 4
    roof = {"kernel": "fattn_bwd_kernel<%d>" % d, "bound": "tensor", "achieved": main_tf,
            "peak": peak_tf, "unit": "TFLOP/s", "frac": main_tf / peak_tf,
            "peak_source": peak_src + " (bf16 burst)",
            "traffic": measured_traffic("fattn_bwd_kernel<%d>" % d) if args.workload == HEADLINE
            else None,
            "algorithmic_bytes": 8 * rows * d * 2 + 2 * rows * 4}
    roof_fwd = {"kernel": "fattn_fwd_kernel<%d>" % d, "bound": "tensor", "achieved": fwd_tf,
                "peak": peak_tf, "unit": "TFLOP/s", "frac": fwd_tf / peak_tf,
                "peak_source": peak_src + " (bf16 burst)",
                "traffic": measured_traffic("fattn_fwd_kernel<%d>" % d) if args.workload == HEADLINE
                else None,
                "algorithmic_bytes": fwd_bytes}

    # the forward's second ceiling: one exponential per visible score against the
    # measured ex2 rate of this GPU
    roof_exp = None
    if do_fwd:
        visible = B * H * (N * (N + 1) / 2.0 if causal else float(N) * N)
        ex2_peak = fattn.ex2_throughput() / 1e12
        exps = visible / (fwd_ms * 1e-3) / 1e12
        roof_exp = {"kernel": "fattn_fwd_kernel<%d>" % d, "bound": "mufu", "achieved": exps,
                    "peak": ex2_peak, "unit": "Texp/s", "frac": exps / ex2_peak,
                    "peak_source": "measured (fattn_ex2_throughput)",
                    "algorithmic_exps": visible}

    # end to end through the C-ABI with host buffers: fattn_fwd_bwd_host copies
    # Q, K, V, dO in from pinned host memory, runs the forward and the backward
    # and copies O, LSE, dQ, dK, dV back, chunk by chunk of heads with the copies
    # and the kernels overlapped
    e2e = None
    if not args.no_e2e and args.passes == "both":
        pin = [x.pin_memory() for x in host]
        outs_h = [torch.empty_like(o, device="cpu").pin_memory(),
                  torch.empty_like(lse, device="cpu").pin_memory(),
                  torch.empty_like(dq, device="cpu").pin_memory(),
                  torch.empty_like(dk, device="cpu").pin_memory(),
                  torch.empty_like(dv, device="cpu").pin_memory()]
        h2d = sum(x.numel() * x.element_size() for x in pin)
        d2h = sum(x.numel() * x.element_size() for x in outs_h)
        hpc = int(args.e2e_chunk)
        e2e_ws_bytes = fattn.fattn_fwd_bwd_host_workspace_bytes(B, H, N, d, hpc)
        e2e_ws = torch.empty(e2e_ws_bytes, dtype=torch.uint8, device=device)

        def e2e_step():
            fattn.fattn_fwd_bwd_host(*pin, *outs_h, B, H, N, d, scale, causal, hpc, e2e_ws,
                                     e2e_ws_bytes, stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(device)
        barrier(world)
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(K):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        assert fattn.fattn_device_error() == 0, "an in-kernel wait timed out"
        e2e_ms = max_over_ranks(a.elapsed_time(b), world, device) / K
        e2e = {"value": job_tflops(world, step_flops, e2e_ms), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "fattn_fwd_bwd_host (pinned host buffers)",
               "heads_per_chunk": hpc if hpc > 0 else "library's choice"}
        del e2e_ws

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == HEADLINE:
        cpu = cpu_baseline(host, scale, causal)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d,
                       "causal": causal, "passes": args.passes,
                       "per_rank": "one full workload per GPU",
                       "l2": "inputs larger than L2 (Q, K, V, dO: %.0f MB each)"
                             % (B * H * N * d * 2 / 1e6)},
            "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak_tf},
            "bwd": {"ms": pre_ms + main_ms + conv_ms, "preprocess_ms": pre_ms,
                    "main_ms": main_ms, "convert_ms": conv_ms,
                    "tflops": f_bwd / ((pre_ms + main_ms + conv_ms) * 1e-3) / 1e12},
            "kernel_times": {"statistic": "median over the timed steps (ms); means beside",
                             "means": means},
            "roofline": roof, "roofline_fwd": roof_fwd, "roofline_fwd_exp": roof_exp,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (int(do_fwd) + 3 * int(do_bwd)) * K,
            "clocks": clk,
        }
        print(json.dumps(_clean(line)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_gpu_varlen(args):
    """Profiling mode for a packed variable-length workload (one GPU): one step is
    fattn_fwd_varlen then fattn_bwd_varlen on all sequences."""
    from online_softmax_08_gb300 import fattn

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = VARLEN_WORKLOADS[args.workload]
    H, d, causal = w["H"], w["d"], w["causal"]
    lens = varlen_lengths(w["B"], w["lo"], w["hi"], w["seed"])
    q, k, v, do, cu = (x.to(device) for x in make_varlen_inputs(lens, H, d, w["seed"], True))
    T, mx, B = int(sum(lens)), max(lens), len(lens)
    scale = default_scale(d)
    f_fwd = sum(4.0 * H * n * n * d * (0.5 if causal else 1.0) for n in lens)
    f_bwd = 2.5 * f_fwd
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fattn.fattn_bwd_workspace_bytes(1, H, T, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    K = args.steps
    evs = [[ev() for _ in range(3)] for _ in range(K)]

    def step(i=None):
        if i is not None:
            evs[i][0].record(stream)
        fattn.fattn_fwd_varlen(q, k, v, o, lse, cu, B, H, mx, T, d, scale, causal, stream)
        if i is not None:
            evs[i][1].record(stream)
        fattn.fattn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu, B, H, mx, T, d, scale, causal,
                               ws, ws_bytes, stream)
        if i is not None:
            evs[i][2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    for e3 in evs:
        for e in e3:
            e.record(stream)
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(device)
    t0, t1 = ev(), ev()
    clocks.region_start()
    t0.record(stream)
    for i in range(K):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks.region_end()
    clk = clocks.stop()
    assert fattn.fattn_device_error() == 0, "an in-kernel wait timed out"
    ms = t0.elapsed_time(t1) / K
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    peak_tf, _, peak_src = peaks()
    fwd_tf, bwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12, f_bwd / (bwd_ms * 1e-3) / 1e12
    line = {
        "metric": "attention fwd/bwd TFLOP/s, packed variable-length batch, d=%d bf16%s"
                  % (d, " causal" if causal else ""),
        "value": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "d": d, "causal": causal,
                   "lengths": "uniform [%d, %d], seed %d" % (w["lo"], w["hi"], w["seed"]),
                   "total_rows": T, "max_seqlen": mx,
                   "l2": "inputs larger than L2 (Q, K, V, dO: %.0f MB each)" % (H * T * d * 2 / 1e6)},
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak_tf},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak_tf},
        "roofline": {"kernel": "fattn_bwd_kernel<%d> (varlen)" % d, "bound": "tensor",
                     "achieved": bwd_tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": bwd_tf / peak_tf, "peak_source": peak_src + " (bf16 burst)",
                     "traffic": None},
        "cpu_baseline": None, "e2e": None, "gpu_launches": 4 * K, "clocks": clk,
    }
    print(json.dumps(_clean(line)), flush=True)
    return 0


def run_gpu_decode(args):
    """Profiling mode for split-KV decoding (one GPU): one step is fattn_decode
    (split forward + merge).  HBM-bound: the roofline is the bytes of K and V
    read once (plus Q, O, LSE) against the measured copy bandwidth."""
    from online_softmax_08_gb300 import fattn

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = DECODE_WORKLOADS[args.workload]
    B, H, Nq, Nkv, d, causal = w["B"], w["H"], w["Nq"], w["Nkv"], w["d"], w["causal"]
    q, k, v = make_inputs(B, H, Nkv, d, w["seed"])
    q = q[:, :, Nkv - Nq:].contiguous()
    q, k, v = q.to(device), k.to(device), v.to(device)
    scale = default_scale(d)
    lib = fattn.load()
    n_splits = int(args.splits)
    S = lib.fattn_decode_splits(B, H, Nq, Nkv, d, n_splits)
    ws = torch.empty(int(lib.fattn_decode_workspace_bytes(B, H, Nq, Nkv, d, n_splits)),
                     dtype=torch.uint8, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    step = lambda: fattn.decode(q, k, v, scale, causal, n_splits, ws, stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.region_start()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks.region_end()
    clk = clocks.stop()
    assert fattn.fattn_device_error() == 0, "an in-kernel wait timed out"
    ms = t0.elapsed_time(t1) / K
    nbytes = (2 * B * H * Nkv * d + 2 * B * H * Nq * d) * 2 + B * H * Nq * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    _, peak_hbm, peak_src = peaks()
    line = {
        "metric": "split-KV decode GB/s (K, V read once), d=%d bf16" % d,
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "Nq": Nq, "Nkv": Nkv, "d": d,
                   "causal": causal, "n_splits": S,
                   "l2": "inputs larger than L2 (K, V: %.0f MB each)" % (B * H * Nkv * d * 2 / 1e6)},
        "roofline": {"kernel": "fattn_fwd_kernel<%d> (split) + merge_kernel" % d, "bound": "hbm",
                     "achieved": gbs, "peak": peak_hbm, "unit": "GB/s", "frac": gbs / peak_hbm,
                     "peak_source": peak_src + " (copy)", "traffic": None,
                     "algorithmic_bytes": nbytes},
        "cpu_baseline": None, "e2e": None, "gpu_launches": 2 * K, "clocks": clk,
    }
    print(json.dumps(_clean(line)), flush=True)
    return 0


def run_gpu_softmax(args):
    """Profiling mode for the row softmax (one GPU): HBM-bound, one read and one
    write of every element (rows fit the shared-memory staging)."""
    from online_softmax_08_gb300 import fattn

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = SOFTMAX_WORKLOADS[args.workload]
    rows, cols = w["rows"], w["cols"]
    x = make_softmax_input(rows, cols, w["seed"]).to(device)
    y = torch.empty_like(x)
    lse = torch.empty((rows,), dtype=torch.float32, device=device)
    lib = fattn.load()
    stream = torch.cuda.current_stream(device)
    step = lambda: fattn._check("fattn_softmax_rows", lib.fattn_softmax_rows(
        x.data_ptr(), y.data_ptr(), lse.data_ptr(), rows, cols, stream.cuda_stream))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.region_start()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks.region_end()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    nbytes = 2 * rows * cols * 4 + rows * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    _, peak_hbm, peak_src = peaks()
    line = {
        "metric": "row softmax GB/s (one read, one write per element), fp32",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "rows": rows, "cols": cols,
                   "l2": "input larger than L2 (%.0f MB)" % (rows * cols * 4 / 1e6)},
        "roofline": {"kernel": "softmax_rows_kernel", "bound": "hbm", "achieved": gbs,
                     "peak": peak_hbm, "unit": "GB/s", "frac": gbs / peak_hbm,
                     "peak_source": peak_src + " (copy)", "traffic": None,
                     "algorithmic_bytes": nbytes},
        "cpu_baseline": None, "e2e": None, "gpu_launches": K, "clocks": clk,
    }
    print(json.dumps(_clean(line)), flush=True)
    return 0


# ------------------------------------------------------------------ host-CPU path

def run_host(args):
    """Profiling mode for the host-CPU flash-style forward (libfattn_host): fp32
    on all host cores, against the fp32 multiply-add peak measured on the same
    threads.  No GPU is used."""
    import numpy as np

    import oracle
    from online_softmax_08_gb300 import fattn_host

    w = HOST_WORKLOADS[args.workload]
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    q, k, v = make_host_inputs(B, H, N, d, w["seed"])
    scale = default_scale(d)
    lib = fattn_host.load()
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float32)
    step = lambda: fattn_host.fattn_host_fwd(q, k, v, o, lse, B, H, N, d, scale, causal)
    for _ in range(args.warmup):
        step()
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    el = time.perf_counter() - t0
    fwd_flops, _ = flops(B, H, N, d, causal)
    ms = el / K * 1e3
    value = fwd_flops / (el / K) / 1e12
    # the public call, with output allocation and argument checks
    t0 = time.perf_counter()
    for _ in range(K):
        fattn_host.forward(q, k, v, scale, causal)
    e2e = fwd_flops * K / (time.perf_counter() - t0) / 1e12
    threads = lib.fattn_host_max_threads()
    peak = lib.fattn_host_fma_peak_gflops(0, 0.5) / 1e3
    line = {
        "metric": "attention fwd TFLOP/s on the host CPU cores, fp32",
        "value": value, "unit": UNIT, "n_gpus": 0, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                   "threads": threads, "device": "host cores (no GPU)"},
        "roofline": {"kernel": "fattn_host_fwd", "bound": "alu", "achieved": value,
                     "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                     "peak_source": "measured: fp32 fused multiply-add loop on the same %d "
                                    "threads" % threads, "traffic": None},
        "cpu_baseline": None, "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0},
        "gpu_launches": 0, "clocks": None,
    }
    if not args.no_cpu_baseline:
        # the fp64 oracle on head 0 of the same inputs, repeated for a few seconds
        qh, kh, vh = (x[:1, :1].astype(np.float64) for x in (q, k, v))
        done, n, t0 = 0.0, 0, time.perf_counter()
        while True:
            oracle.attention_fwd(qh, kh, vh, scale, causal)
            done += flops(1, 1, N, d, causal)[0]
            n += 1
            t = time.perf_counter() - t0
            if t >= 5.0:
                break
        line["cpu_baseline"] = {"value": done / t / 1e12, "unit": UNIT,
                                "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": "fp64 oracle forward of head 0 (N=%d), %d times "
                                          "(%.1f s)" % (N, n, t)}
    print(json.dumps(_clean(line)), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=sorted(WORKLOADS) + sorted(VARLEN_WORKLOADS) + sorted(DECODE_WORKLOADS)
                    + sorted(SOFTMAX_WORKLOADS) + sorted(HOST_WORKLOADS),
                    help="profiling only: the benchmark's workload is the default")
    ap.add_argument("--pass", dest="passes", default="both", choices=["both", "fwd", "bwd"],
                    help="profiling only: time one pass; a benchmark step is both")
    ap.add_argument("--splits", default=0, help="decode workloads: key ranges (0 = automatic)")
    ap.add_argument("--causal", default="default", choices=["default", "yes", "no"],
                    help="profiling only: the masking mode of a fixed-shape workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunk", default=0,
                    help="heads per chunk of the end-to-end leg (0 = the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in VARLEN_WORKLOADS:
        return run_gpu_varlen(args)
    if args.workload in DECODE_WORKLOADS:
        return run_gpu_decode(args)
    if args.workload in SOFTMAX_WORKLOADS:
        return run_gpu_softmax(args)
    if args.workload in HOST_WORKLOADS:
        return run_host(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
