"""Benchmark: attention forward + backward TFLOP/s on GB300 through the C ABI.

One step = the whole hot path over one batch: fa_fwd, then the three backward stages
(fa_bwd_preprocess, fa_bwd_main, fa_bwd_dq_convert).  The line also carries a split-KV
decode measurement (``decode``: fa_decode over a 1.07 GB key/value cache, HBM-bound).  Default workload: the causal LM
shape B=8, H=16, N=4096, d=128, bf16 (FLOPs: forward 4·B·H·N²·d, backward 2.5x, halved
for causal).  Inputs are larger than L2 (each [B,H,N,d] tensor is 134 MB).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line on rank 0.  ``--impl reference`` times the fp64 CPU oracle (there is no reference code
to run, so the oracle is the reference arm) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_tiled_attention_07_gb300.inputs import (  # noqa: E402
    DECODE_WORKLOADS,
    WORKLOADS,
    Workload,
    attention_flops,
    make_decode_inputs,
    make_inputs,
)

METRIC = "attention fwd/bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "causal_lm_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def source_digest():
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "exact_tiled_attention_07_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key, workload):
    """DRAM bytes per launch of a kernel on a workload from a committed ncu summary, if the
    summary was taken on the current sources (else None)."""
    digest = source_digest()
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(p) as f:
            for line in f:
                # machine-readable line: "traffic: <kernel_key> <workload> <bytes_per_launch> sources=<digest>"
                if line.startswith("traffic:"):
                    parts = line.split()
                    if (len(parts) >= 5 and parts[1] == kernel_key and parts[2] == workload
                            and parts[4] == f"sources={digest}"):
                        return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms; summary() keeps the timed window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons over samples inside [t0, t1] (wall clock)."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for ts, ln in self.lines:
            cols = [c.strip() for c in ln.split(",")]
            if len(cols) < 9:
                continue
            try:
                parsed.append((ts, float(cols[1]), float(cols[2]), cols[5:9]))
            except ValueError:
                continue
        window = [p for p in parsed if t0 is None or (t0 <= p[0] <= t1 + 0.1)]
        note = "samples inside the timed region"
        if not window and parsed:
            window = parsed
            note = "no sample fell inside the timed region; all samples of the run"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({nm for p in window for nm, v in zip(names, p[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(p[1] for p in window), "sm_max_mhz": max(p[2] for p in window),
                "reasons": reasons, "samples": len(window), "note": note}


# Dense 16-bit tensor-core work per SM per clock: one 128 x N x 16 MMA every N / 2 cycles, i.e.
# 4096 multiply-adds (the published dense bf16 rate, 2.25 PFLOP/s on 148 SMs at about 1.86 GHz).
TENSOR_FLOP_PER_SM_CLOCK = 8192
# A timed region shorter than this is a burst: the kernel is compared with the burst peak.
BURST_REGION_S = 1.0


def sm_clock_mhz(before, after):
    """Per-SM mean clock (MHz) between two fa_sm_clock_sample readings (rows of SM id, cycle
    counter, global timer in ns): for each SM seen in both, cycles elapsed over ns elapsed."""
    first = {int(r[0]): (int(r[1]), int(r[2])) for r in before}
    out = []
    for r in after:
        sm = int(r[0])
        if sm in first and int(r[2]) > first[sm][1]:
            out.append(1e3 * (int(r[1]) - first[sm][0]) / (int(r[2]) - first[sm][1]))
    return out


def peak_for_region(peaks, region_s):
    """(peak TFLOP/s, which one): the burst cuBLAS figure for a region shorter than
    BURST_REGION_S, the sustained (seconds-long, power-capped) figure otherwise."""
    if region_s < BURST_REGION_S:
        return float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])), "bf16_tflops (burst)"
    return float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])), \
        "bf16_tflops_sustained (seconds-long region)"


def tensor_peak_at_clock(sm_mhz, n_sm):
    """Dense 16-bit tensor peak (TFLOP/s) of n_sm SMs at the given clock."""
    return n_sm * TENSOR_FLOP_PER_SM_CLOCK * sm_mhz * 1e6 / 1e12


# ---------------------------------------------------------------------------
# CPU oracle arm (the reference arm) and the cpu_baseline leg
# ---------------------------------------------------------------------------


def oracle_heads(w: Workload, target_s: float, max_heads: int):
    """Run the fp64 oracle (forward + backward) on whole heads until ~target_s of compute.

    Returns (heads, seconds of oracle compute); input generation is not timed.
    """
    import oracle
    from exact_tiled_attention_07_gb300.inputs import to_float64

    one = w.with_shape(B=1, H=1)
    heads, elapsed = 0, 0.0
    while heads < max_heads and (heads == 0 or elapsed < target_s):
        x = make_inputs(one.with_shape(seed=w.seed + heads))
        x64 = {k: to_float64(v, w.dtype) for k, v in x.items()}
        t0 = time.perf_counter()
        oracle.attn_fwd64(x64["q"], x64["k"], x64["v"], w.scale, w.causal)
        if not w.fwd_only:
            oracle.attn_bwd64(x64["q"], x64["k"], x64["v"], x64["do"], w.scale, w.causal)
        elapsed += time.perf_counter() - t0
        heads += 1
    return heads, elapsed


def oracle_sample(w: Workload, target_s: float = 12.0, max_heads: int = 64):
    """The cpu_baseline leg: the oracle as it stands, on whole heads of the workload (~target_s)."""
    heads, elapsed = oracle_heads(w, target_s, max_heads)
    pass_ = "fwd" if w.fwd_only else "fwd+bwd"
    flops = attention_flops(1, 1, w.N, w.d, w.causal, pass_) * heads
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} heads ({w.N}x{w.d}, {pass_}), numpy fp64, {elapsed:.1f} s"}


def run_reference(args, w: Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_heads(w, 0.0, 1)
    times = [oracle_heads(w, 0.0, 1)[1] for _ in range(args.steps)]
    pass_ = "fwd" if w.fwd_only else "fwd+bwd"
    flops = attention_flops(1, 1, w.N, w.d, w.causal, pass_)
    value = flops * len(times) / sum(times) / 1e12
    cpu = {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
           "sample": f"1 of {w.B * w.H} heads per step ({w.N}x{w.d}, {pass_}), numpy fp64"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w), "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w: Workload):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype, "causal": w.causal,
            "passes": "fwd" if w.fwd_only else "fwd+bwd",
            "l2": l2_note(w)}


def l2_note(w: Workload) -> str:
    """What keeps L2 from serving a step's inputs from the previous step (no flush is done)."""
    e = 4 if w.dtype == "fp32" else 2
    ins = (w.B * w.H * w.N * w.d + 2 * w.B * w.kv_heads * w.N * w.d) * e  # Q, K, V
    if not w.fwd_only:
        ins += w.B * w.H * w.N * w.d * e  # dO
    if ins > 129e6:
        return f"inputs of {ins / 1e6:.0f} MB per step, larger than the 129 MB L2 (no flush)"
    return f"inputs of {ins / 1e6:.1f} MB per step fit in L2 (no flush)"


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def shard_workload(w: Workload, rank: int) -> Workload:
    """Rank r's independent shard: the same shape, its own seed (weak scaling, no exchange)."""
    return w.with_shape(seed=w.seed + 1000 * rank)


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest of each rank's value (one all-reduce of a scalar); x itself on one process."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the work all ranks did in one step over the slowest rank's step time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def _dev_tensor(stored, dtype, device):
    import torch

    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(stored).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(stored))
    return t.pin_memory().to(device, non_blocking=False), t.pin_memory()


def measure_decode(binding, device, peaks, peak_src, reps=50):
    """Split-KV decode over a key/value cache larger than L2: HBM bytes per second of one
    fa_decode call (the partial kernel and the merge), against the measured HBM bandwidth."""
    import torch

    w = DECODE_WORKLOADS["decode_gqa_bf16"]
    x = make_decode_inputs(w)
    q, k, v = (_dev_tensor(x[n], w.dtype, device)[0] for n in ("q", "k", "v"))
    del x
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=device)
    nbytes = binding.fa_decode_workspace_size(w.B, w.H, w.Hkv, w.Nq, w.Nk, w.d, 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)

    def call():
        binding.fa_decode(q, k, v, o, lse, w.scale, 0, ws)

    for _ in range(5):
        call()
    binding.fa_check_device_error()
    stream = torch.cuda.current_stream()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)  # the first calls are queued before the start event fires
    a_.record(stream)
    for _ in range(reps):
        call()
    b_.record(stream)
    torch.cuda.synchronize()
    binding.fa_check_device_error()
    us = a_.elapsed_time(b_) / reps * 1e3
    gbs = w.bytes_moved() / (us * 1e-6) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
            "dtype": w.dtype, "us_per_call": us, "calls": reps, "launches_per_call": 2,
            "roofline": {"kernel": "decode_tc_kernel + decode_merge", "bound": "hbm", "achieved": gbs,
                         "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": profiled_traffic("decode_tc", w.name),
                         "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)",
                         "algorithmic_bytes": w.bytes_moved()},
            "l2": "cache of 1.07 GB, larger than L2 (no flush)"}


def run_gpu(args, w: Workload):
    import torch

    from exact_tiled_attention_07_gb300 import binding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load_library()

    # every rank owns an independent shard of the same shape (weak scaling, no exchange)
    x = make_inputs(shard_workload(w, rank), with_do=not w.fwd_only)
    dev, pinned = {}, {}
    for k_, v_ in x.items():
        dev[k_], pinned[k_] = _dev_tensor(v_, w.dtype, device)
    del x
    q, k, v = dev["q"], dev["k"], dev["v"]
    do = dev.get("do")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    if not w.fwd_only:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    scale, causal = w.scale, w.causal
    names = ["fwd"] if w.fwd_only else ["fwd", "bwd_pre", "bwd_main", "bwd_dq_convert"]

    def launch(i, causal_=causal):
        if i == 0:
            binding.fa_fwd(q, k, v, o, lse, scale, causal_)
        elif i == 1:
            binding.fa_bwd_preprocess(o, do, lse, ws)
        elif i == 2:
            binding.fa_bwd_main(q, k, v, do, dk, dv, ws, scale, causal_)
        else:
            binding.fa_bwd_dq_convert(ws, dq, scale)

    def step(evs=None):
        for i in range(len(names)):
            if evs is not None:
                evs[i].record(stream)
            launch(i)
        if evs is not None:
            evs[len(names)].record(stream)

    for _ in range(args.warmup):
        step()
    binding.fa_check_device_error()

    # ---------------- timed region: K steps, per-kernel events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # every SM's cycle counter read just before and just after the timed region (outside its
    # events): each SM's mean clock over exactly the timed steps
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    smc = [torch.zeros(3 * n_sm, dtype=torch.int64, device=device) for _ in range(2)]
    with ClockSampler(local) as clocks:
        time.sleep(0.5)  # let the sampler start
        wall0 = time.time()
        binding.fa_sm_clock_sample(smc[0], stream)
        t_start.record(stream)
        for s_ in range(args.steps):
            step(ev[s_])
        t_end.record(stream)
        binding.fa_sm_clock_sample(smc[1], stream)
        torch.cuda.synchronize()
        wall1 = time.time()
    if dist:
        dist.barrier()
    binding.fa_check_device_error()
    total_ms = t_start.elapsed_time(t_end)
    per_kernel = {nm: sum(ev[s_][i].elapsed_time(ev[s_][i + 1]) for s_ in range(args.steps)) / args.steps
                  for i, nm in enumerate(names)}
    total_ms = max_over_ranks(total_ms, dist, device)
    ms_per_step = total_ms / args.steps
    pass_ = "fwd" if w.fwd_only else "fwd+bwd"
    flops_rank = attention_flops(w.B, w.H, w.N, w.d, w.causal, pass_)
    value = aggregate_tflops(flops_rank, world, ms_per_step)

    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    region_s = total_ms * 1e-3
    peak, peak_kind = peak_for_region(peaks, region_s)
    mhz = sm_clock_mhz(smc[0].cpu().numpy().reshape(-1, 3), smc[1].cpu().numpy().reshape(-1, 3))
    sm_mhz_dev = statistics.median(mhz) if mhz else None

    # ---------------- roofline of the dominant kernel
    kflops = {"fwd": attention_flops(w.B, w.H, w.N, w.d, w.causal, "fwd"),
              "bwd_main": attention_flops(w.B, w.H, w.N, w.d, w.causal, "bwd")}
    dom = max((nm for nm in per_kernel if nm in kflops), key=lambda nm: per_kernel[nm])
    achieved = kflops[dom] / (per_kernel[dom] * 1e-3) / 1e12
    traffic = profiled_traffic(dom, w.name)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} {peak_kind}: the timed region lasted {region_s:.3f} s",
                "share_of_step": per_kernel[dom] / ms_per_step}
    if sm_mhz_dev:
        at_clock = tensor_peak_at_clock(sm_mhz_dev, n_sm)
        roofline.update({"frac_at_clock": achieved / at_clock, "peak_at_clock": at_clock,
                         "peak_at_clock_source": f"{n_sm} SMs x {TENSOR_FLOP_PER_SM_CLOCK} FLOP/clock x "
                                                 f"{sm_mhz_dev:.0f} MHz (median SM clock over the timed region, "
                                                 f"from each SM's cycle counter)"})

    # ---------------- end to end: pinned host buffers -> device, the C-ABI calls, results -> host
    def measure_e2e():
        h2d = sum(pinned[k_].numel() * pinned[k_].element_size() for k_ in pinned)
        outs = [o, lse] + ([] if w.fwd_only else [dq, dk, dv])
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        d2h = sum(t.numel() * t.element_size() for t in outs)
        ins = [(dev[k_], pinned[k_]) for k_ in pinned]
        if not w.fwd_only:
            # one C-ABI call over the host buffers: chunks of heads copied in, computed and copied
            # out on the library's streams, overlapping the copies of one chunk with its neighbours'
            # computation
            ws_host = torch.empty(binding.fa_fwd_bwd_host_workspace_size(w.B, w.H, w.H, w.N, w.d, q.dtype,
                                                                         args.e2e_chunk),
                                  dtype=torch.uint8, device=device)

            def e2e_step():
                binding.fa_fwd_bwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["do"], *host_out, ws_host, scale,
                                        causal, args.e2e_chunk, stream)
        else:
            def e2e_step():
                for d_, h_ in ins:
                    d_.copy_(h_, non_blocking=True)
                step()
                for h_, d_ in zip(host_out, outs):
                    h_.copy_(d_, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e_s.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e_e.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e_s.elapsed_time(e_e) / args.steps
        e2e_ms = max_over_ranks(e2e_ms, dist, device)
        e2e = {"value": aggregate_tflops(flops_rank, world, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "call": "fa_fwd_bwd_host" if not w.fwd_only else "copies + fa_fwd",
               "chunk_kv_heads": args.e2e_chunk if not w.fwd_only else None}
        return e2e

    e2e = None if args.no_e2e else measure_e2e()

    # ---------------- per-pass figures, including the non-causal variant of the same shape
    targets = None
    if not args.no_targets:
        targets = {}
        variants = [(causal, "causal" if causal else "noncausal")]
        if causal:
            variants.append((False, "noncausal"))
        for cz, tag in variants:
            passes = [("fwd", [0])] + ([] if w.fwd_only else [("bwd", [1, 2, 3])])
            for pname, idxs in passes:
                reps = max(3, min(args.steps, 10))
                for _ in range(2):
                    for i in idxs:
                        launch(i, cz)
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                for _ in range(reps):
                    for i in idxs:
                        launch(i, cz)
                b_.record(stream)
                torch.cuda.synchronize()
                ms = a_.elapsed_time(b_) / reps
                fl = attention_flops(w.B, w.H, w.N, w.d, cz, pname)
                tf = fl / (ms * 1e-3) / 1e12
                targets[f"{tag}_{pname}"] = {"ms": ms, "tflops": tf, "pct_of_burst_peak": 100 * tf / peak_burst,
                                             "pct_of_sustained_peak": 100 * tf / peak_sus}
        if w.d == 128 and w.dtype != "fp32":
            # FP8 forward on block-quantised copies of the same inputs (quantised once, untimed);
            # its peak is the bf16 peak x 2 (the nominal dense fp8 / bf16 ratio)
            q8, qs = binding.quantize_fp8(q)
            k8, ks = binding.quantize_fp8(k)
            v8, vs = binding.quantize_fp8(v)
            o8 = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
            for cz, tag in variants:
                reps = max(3, min(args.steps, 10))

                def fp8_call():
                    binding.fa_fwd_fp8(q8, k8, v8, qs, ks, vs, o8, lse, scale, cz)

                for _ in range(2):
                    fp8_call()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                for _ in range(reps):
                    fp8_call()
                b_.record(stream)
                torch.cuda.synchronize()
                ms = a_.elapsed_time(b_) / reps
                tf = attention_flops(w.B, w.H, w.N, w.d, cz, "fwd") / (ms * 1e-3) / 1e12
                targets[f"{tag}_fwd_fp8"] = {"ms": ms, "tflops": tf, "pct_of_fp8_burst_peak": 100 * tf / (2 * peak_burst),
                                             "pct_of_fp8_sustained_peak": 100 * tf / (2 * peak_sus),
                                             "fp8_peak": "derived: 2 x the measured bf16 peak (the nominal dense "
                                                         "fp8 / bf16 ratio); no fp8 peak was measured"}
            reps = max(3, min(args.steps, 10))
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            for _ in range(reps):
                binding.fa_quantize_fp8(q, q8, qs)
            b_.record(stream)
            torch.cuda.synchronize()
            ms = a_.elapsed_time(b_) / reps
            qbytes = q.numel() * (q.element_size() + 1) + qs.numel() * 4
            targets["quantize_fp8"] = {"ms": ms, "gbs": qbytes / (ms * 1e-3) / 1e9,
                                       "frac_of_hbm": qbytes / (ms * 1e-3) / 1e9 / float(peaks.get("hbm_gbs", 6800.0))}
            del q8, k8, v8, o8
        binding.fa_check_device_error()

    # the other full-size workloads of the pages (same step, same timing): GPT-2-medium shape
    # (fp16, d = 64) and the long causal sequence (bf16, d = 64)
    others = None
    if not args.no_targets and rank == 0:
        others = {}
        for wname in ("gpt2m_fp16", "long_causal_bf16", "hd256_bf16"):
            ow = WORKLOADS[wname]
            # the head-dimension-256 workload is forward only; its backward is timed as an
            # extra leg ("bwd_extra"), not part of the workload's passes
            with_bwd = not ow.fwd_only or ow.d == 256
            ox = make_inputs(ow, with_do=with_bwd)
            od = {k_: _dev_tensor(v_, ow.dtype, device)[0] for k_, v_ in ox.items()}
            del ox
            oo = torch.empty_like(od["q"])
            ol = torch.empty((ow.B, ow.H, ow.N), dtype=torch.float32, device=device)
            odq = odk = odv = ows = None
            if with_bwd:
                odq, odk, odv = torch.empty_like(od["q"]), torch.empty_like(od["k"]), torch.empty_like(od["v"])
                ows = torch.empty(binding.fa_bwd_workspace_size(ow.B, ow.H, ow.N, ow.d), dtype=torch.uint8,
                                  device=device)

            def ofwd():
                binding.fa_fwd(od["q"], od["k"], od["v"], oo, ol, ow.scale, ow.causal)

            def obwd():
                binding.fa_bwd(od["q"], od["k"], od["v"], oo, od["do"], ol, odq, odk, odv, ows, ow.scale, ow.causal)

            entry = {"config": workload_config(ow)}
            reps = max(3, min(args.steps, 10))
            legs = ((("fwd", (ofwd,)), ("bwd_extra", (obwd,))) if ow.fwd_only
                    else (("fwd", (ofwd,)), ("bwd", (obwd,)), ("fwd+bwd", (ofwd, obwd))))
            for pname, fns in legs:
                for _ in range(2):
                    for fn in fns:
                        fn()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                for _ in range(reps):
                    for fn in fns:
                        fn()
                b_.record(stream)
                torch.cuda.synchronize()
                ms = a_.elapsed_time(b_) / reps
                tf = attention_flops(ow.B, ow.H, ow.N, ow.d, ow.causal, "bwd" if pname == "bwd_extra" else pname)
                tf /= (ms * 1e-3) * 1e12
                entry[pname] = {"ms": ms, "tflops": tf, "pct_of_burst_peak": 100 * tf / peak_burst,
                                "pct_of_sustained_peak": 100 * tf / peak_sus}
                if pname == "bwd_extra":
                    entry[pname]["note"] = "backward (3 kernels) of the same inputs; not a pass of this workload"
            if ow.d in (64, 128, 256) and ow.dtype != "fp32":
                # FP8 forward on block-quantised copies of the same inputs (quantised once, untimed)
                (q8, qs), (k8, ks), (v8, vs) = (binding.quantize_fp8(od[n_]) for n_ in ("q", "k", "v"))

                def ofp8():
                    binding.fa_fwd_fp8(q8, k8, v8, qs, ks, vs, oo, ol, ow.scale, ow.causal)

                for _ in range(2):
                    ofp8()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                for _ in range(reps):
                    ofp8()
                b_.record(stream)
                torch.cuda.synchronize()
                ms = a_.elapsed_time(b_) / reps
                tf = attention_flops(ow.B, ow.H, ow.N, ow.d, ow.causal, "fwd") / (ms * 1e-3) / 1e12
                entry["fwd_fp8"] = {"ms": ms, "tflops": tf, "pct_of_fp8_burst_peak": 100 * tf / (2 * peak_burst),
                                    "fp8_peak": "derived: 2 x the measured bf16 burst (the nominal dense fp8 / bf16 ratio)"}
                del q8, k8, v8
            others[wname] = entry
            del od, oo, ol, odq, odk, odv, ows
        binding.fa_check_device_error()

    decode = None
    if not args.no_decode:
        decode = measure_decode(binding, device, peaks, peak_src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(w)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": workload_config(w),
                "pct_of_peak": {"sustained": 100 * value / world / peak_sus, "burst": 100 * value / world / peak_burst,
                                "at_clock": (100 * value / world / tensor_peak_at_clock(sm_mhz_dev, n_sm)
                                             if sm_mhz_dev else None),
                                "source": peak_src},
                "kernels_ms": per_kernel, "gpu_launches": len(names) * args.steps, "roofline": roofline,
                "e2e": e2e, "clocks": dict(clocks.summary(wall0, wall1), sm_mhz_device=sm_mhz_dev,
                                           sm_mhz_device_range=[min(mhz), max(mhz)] if mhz else None,
                                           sm_seen=len(mhz)),
                "cpu_baseline": cpu, "targets": targets,
                "other_workloads": others, "decode": decode}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the split-KV decode measurement")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer measurement")
    ap.add_argument("--e2e-chunk", type=int, default=0,
                    help="key/value heads per chunk of the end-to-end host-buffer call (0: automatic)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return
    run_gpu(args, w)


if __name__ == "__main__":
    main()
