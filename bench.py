"""Throughput benchmark of the exact-attention hot path on GB300.

Default workload: the dense non-causal MHA configuration B=2, H=16, N=8192,
D=128 (bf16 Q/K/V/dO iid N(0,1) from seed 0, scale = 1/sqrt(D)).  One step is
one pass of the whole hot path over that batch: the forward (O, LSE) and,
when the backward is built, the LSE-recompute backward (dQ, dK, dV).

FLOP convention: forward 4*B*Hq*N^2*D (halved when causal), backward 2.5x the
forward.  `value` is TFLOPS of the step (all ranks), timed with CUDA events on
the launch stream between barriers + device synchronisation.  The default
workload's inputs (256 MiB) exceed the 129 MB L2, so its steps run back to
back; a workload whose inputs fit in L2 is timed step by step instead, with a
256 MiB buffer written before every step (outside the timed spans).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference   # the fp64 CPU oracle on a bounded sample

Prints ONE JSON line on rank 0.
"""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (bf16, fwd & fwd+bwd) and % of GB300 tensor-core peak"
L2_BYTES = 129 * 10**6  # GB300 L2
UNIT = "TFLOPS"

WORKLOADS = {
    # name: (B, Hq, Hkv, N, D, causal, description)
    "dense_b2_h16_n8192_d128": (2, 16, 16, 8192, 128, False,
                                "dense non-causal MHA, B=2 H=16 N=8192 D=128"),
    "dense_b4_h16_n4096_d128": (4, 16, 16, 4096, 128, False,
                                "dense non-causal MHA, B=4 H=16 N=4096 D=128"),
    "dense_b1_h16_n16384_d128": (1, 16, 16, 16384, 128, False,
                                 "dense non-causal MHA, B=1 H=16 N=16384 D=128"),
    "causal_b1_h16_n4096_d64": (1, 16, 16, 4096, 64, True,
                                "causal MHA training step, B=1 H=16 N=4096 D=64"),
    "causal_gqa_b1_h8_2_n4096_d128": (1, 8, 2, 4096, 128, True,
                                      "causal GQA, B=1 Hq=8 Hkv=2 N=4096 D=128"),
    "causal_b1_h16_n2048_d64": (1, 16, 16, 2048, 64, True,
                                "causal MHA, B=1 H=16 N=2048 D=64"),
    "causal_b1_h16_n2000_d64": (1, 16, 16, 2000, 64, True,
                                "causal MHA, B=1 H=16 N=2000 D=64 (ragged last tile)"),
    "dense_b1_h2_n256_d64": (1, 2, 2, 256, 64, False,
                             "non-causal MHA, B=1 H=2 N=256 D=64"),
    "dense_b2_h16_n8192_d64": (2, 16, 16, 8192, 64, False,
                               "dense non-causal MHA, B=2 H=16 N=8192 D=64"),
    "causal_b2_h16_n8192_d128": (2, 16, 16, 8192, 128, True,
                                 "causal MHA, B=2 H=16 N=8192 D=128"),
}
DEFAULT_WORKLOAD = "dense_b2_h16_n8192_d128"


def fwd_flops(B, Hq, N, D, causal):
    f = 4.0 * B * Hq * N * N * D
    return f / 2 if causal else f


def _measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    return 1900.0, 1700.0, "fallback"


def _measured_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _kernel_source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flash_exact_attention_gb300", "csrc")
    for n in sorted(names):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


NYS_SOURCES = ["nys_kernel.cuh", "ptx.cuh", "nys.cu", "nys_d128.cu", "nys_d64.cu"]
FWD_SOURCES = ["fwd_kernel.cuh", "ptx.cuh", "fwd_launch.cuh", "fwd_d128.cu", "fwd_d64.cu"]
BWD_SOURCES = ["bwd_kernel.cuh", "ptx.cuh", "bwd_launch.cuh", "bwd.cu", "bwd_d128.cu",
               "bwd_d64.cu"]


def _recorded_traffic(kernel, workload, src_hash):
    """DRAM bytes per launch from profiles/dram_traffic.md, if taken on this source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[2] == src_hash:
            try:
                return float(cells[3])
            except ValueError:
                return None
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        # nvidia-smi's start-up briefly stalls the device; let it pass before timing.
        time.sleep(1.5)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                smax = float(c[2])
            except ValueError:
                continue
            for name, val in zip(names, c[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings: the slowest rank sets the job time."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world_size, flops_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank does one step of the same size (weak scaling)."""
    return world_size * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def rank_seed(seed, rank):
    """Each rank draws its own batch: the replicas share no data and no collective."""
    return seed + rank


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_native(args):
    import numpy as np
    import torch

    from flash_exact_attention_gb300 import binding
    from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    B, Hq, Hkv, N, D, causal, desc = WORKLOADS[args.workload]
    scale = scale_for(D)
    has_bwd = STEP_INCLUDES_BWD

    x = make_inputs(B, Hq, Hkv, N, D, seed=rank_seed(args.seed, rank), with_do=True)
    host = {n: to_torch_bf16(a).pin_memory() for n, a in x.items()}
    dev = {n: t.to("cuda") for n, t in host.items()}
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def fwd():
        st = binding.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, sh)
        if st:
            raise binding.AttnError(st, "attn_fwd")

    def bwd():
        st = binding.attn_bwd(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, sh, do, dq, dk,
                              dv)
        if st:
            raise binding.AttnError(st, "attn_bwd")

    def step():
        fwd()
        if has_bwd:
            bwd()

    launches_per_step = 1 + (BWD_LAUNCHES if has_bwd else 0)
    ff = fwd_flops(B, Hq, N, D, causal)
    step_flops = ff * (3.5 if has_bwd else 1.0)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- warm-up
    for _ in range(args.warmup):
        step()
    barrier()
    st = binding.attn_device_status(sh)
    if st:
        raise binding.AttnError(st, "warm-up")

    # Inputs that fit in L2 would be served from it by the next step: scrub L2
    # (write a buffer larger than it) before every timed step, timing each step
    # with its own events so the scrub stays outside the measurement.
    in_bytes = sum(host[n].numel() * host[n].element_size() for n in ("q", "k", "v", "do"))
    scrub_l2 = in_bytes < L2_BYTES
    scrub = torch.empty(256 * 2**20, dtype=torch.uint8, device="cuda") if scrub_l2 else None

    def timed_steps(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            scrub.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        barrier()
        return sum(a.elapsed_time(b) for a, b in evs)

    def back_to_back():
        """Whole steps, then forward calls, then backward calls, each run back
        to back between one pair of events on the launch stream."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            fwd()
        f1.record(stream)
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        if has_bwd:
            b0.record(stream)
            for _ in range(args.steps):
                bwd()
            b1.record(stream)
        barrier()
        return (e0.elapsed_time(e1), f0.elapsed_time(f1),
                b0.elapsed_time(b1) if has_bwd else 0.0)

    # ---- timed region: CUDA events on the launch stream, clocks sampled meanwhile
    with ClockSampler(local) as clk:
        barrier()
        if scrub_l2:
            ms_total = timed_steps(step)
            ms_fwd = timed_steps(fwd)
            ms_bwd = timed_steps(bwd) if has_bwd else 0.0
        else:
            ms_total, ms_fwd, ms_bwd = back_to_back()
    st = binding.attn_device_status(sh)
    if st:
        raise binding.AttnError(st, "timed region")

    ms_step = ms_total / args.steps
    ms_fwd_launch = ms_fwd / args.steps
    ms_bwd_call = ms_bwd / args.steps
    ms_step, ms_fwd_launch, ms_bwd_call = max_over_ranks(
        [ms_step, ms_fwd_launch, ms_bwd_call], dist, "cuda")
    value = job_tflops(ws, step_flops, ms_step)
    fwd_tflops = ff / (ms_fwd_launch * 1e-3) / 1e12
    bwd_tflops = 2.5 * ff / (ms_bwd_call * 1e-3) / 1e12 if has_bwd else None

    # ---- end to end through the C ABI from pinned host buffers: every step copies
    # its inputs in and its results out.  As a training or serving loop would, the
    # copies run on their own streams (host->device and device->host engines) and
    # overlap the neighbouring steps' kernels, with two device buffer sets.
    out_names = ["o", "lse"] + (["dq", "dk", "dv"] if has_bwd else [])
    outs = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    host_out = {n: torch.empty(outs[n].shape, dtype=outs[n].dtype, pin_memory=True)
                for n in out_names}
    in_names = ["q", "k", "v"] + (["do"] if has_bwd else [])
    h2d = sum(host[n].numel() * host[n].element_size() for n in in_names)
    d2h = sum(host_out[n].numel() * host_out[n].element_size() for n in out_names)
    # Steps per pass: each pass starts with the first step's host->device copy and
    # ends with the last step's device->host copy, neither overlapped; 60 steps
    # amortise them as a training loop does (each pass still pays both).
    e2e_steps = max(3, min(args.steps, 60))
    bufs = [dict(dev, **outs), {n: torch.empty_like(t) for n, t in dict(dev, **outs).items()}]

    # Three streams of their own (none is the legacy default stream, which would
    # serialise with the others).
    comp_stream, h2d_stream, d2h_stream = (torch.cuda.Stream(), torch.cuda.Stream(),
                                           torch.cuda.Stream())
    csh = comp_stream.cuda_stream

    def step_on(b):
        st = binding.attn_fwd(b["q"], b["k"], b["v"], b["o"], b["lse"], B, Hq, Hkv, N, D, causal,
                              scale, csh)
        if st:
            raise binding.AttnError(st, "attn_fwd")
        if has_bwd:
            st = binding.attn_bwd(b["q"], b["k"], b["v"], b["o"], b["lse"], B, Hq, Hkv, N, D,
                                  causal, scale, csh, b["do"], b["dq"], b["dk"], b["dv"])
            if st:
                raise binding.AttnError(st, "attn_bwd")

    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    def e2e_pass():
        """e2e_steps pipelined steps; returns ms per step (CUDA events)."""
        barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(comp_stream)
        h2d_stream.wait_event(g0)
        for i in range(e2e_steps):
            b = i % 2
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(ev_comp[b])  # step i-2 is done reading set b
                for n in in_names:
                    bufs[b][n].copy_(host[n], non_blocking=True)
                ev_in[b].record(h2d_stream)
            comp_stream.wait_event(ev_in[b])
            if i >= 2:
                comp_stream.wait_event(ev_out[b])  # step i-2's results in set b are copied out
            step_on(bufs[b])
            ev_comp[b].record(comp_stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_comp[b])
                for n in out_names:
                    host_out[n].copy_(bufs[b][n], non_blocking=True)
                ev_out[b].record(d2h_stream)
        g1.record(d2h_stream)
        barrier()
        return g0.elapsed_time(g1) / e2e_steps

    e2e_pass()  # untimed: first use of the second buffer set and of the host buffers
    e2e_runs = sorted(e2e_pass() for _ in range(3))
    ms_e2e = e2e_runs[1]  # median of three timed passes
    st = binding.attn_device_status(csh)
    if st:
        raise binding.AttnError(st, "end-to-end leg")
    ms_e2e = max_over_ranks([ms_e2e], dist, "cuda")[0]
    e2e_value = job_tflops(ws, step_flops, ms_e2e)

    peak_burst, peak_sust, peak_src = _measured_peaks()
    peak_note = ("%s bf16 burst (MEASURED_PEAKS.json)" % peak_src if peak_src == "measured"
                 else "fallback 1.9 PFLOP/s")
    tag = "%d,%s" % (D, "causal" if causal else "noncausal")

    def roof(kernel, sources, tflops, flops):
        h = _kernel_source_hash(sources)
        return {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak_burst,
                "unit": "TFLOP/s", "frac": round(tflops / peak_burst, 4),
                "traffic": _recorded_traffic(kernel, args.workload, h), "kernel": kernel,
                "peak_source": peak_note, "frac_of_sustained": round(tflops / peak_sust, 4),
                "algorithmic_flops_per_launch": flops, "source_hash": h}

    roof_fwd = roof("fwd_kernel<%s>" % tag, FWD_SOURCES, fwd_tflops, ff)
    if has_bwd:
        # The backward call (preprocess + main + postprocess, timed together) is
        # the dominant part of the step; its FLOPs are the main kernel's.
        roofline = roof("bwd_kernel<%s>" % tag, BWD_SOURCES, bwd_tflops, 2.5 * ff)
        roofline["timed_as"] = "whole attn_bwd call (3 launches)"
    else:
        roofline = roof_fwd
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic iid N(0,1) bf16 from numpy seed %d (+rank)" % args.seed,
        "config": {"workload": desc, "name": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv,
                   "N": N, "D": D, "causal": causal,
                   "step": "fwd+bwd" if has_bwd else "fwd (backward not built)",
                   "parallelism": "replicas" if ws == 1 else "dp%d (independent batches)" % ws,
                   "l2": ("flushed: a 256 MiB buffer written before every timed step (inputs "
                          "%.0f MiB fit in the 129 MB L2; one pair of events per step)"
                          % (in_bytes / 2**20)) if scrub_l2 else
                         ("no flush: per-step inputs %.0f MiB exceed the 129 MB L2"
                          % (in_bytes / 2**20))},
        "fwd_tflops": round(fwd_tflops, 1),
        "fwd_pct_of_peak": round(100 * fwd_tflops / peak_burst, 2),
        "bwd_tflops": round(bwd_tflops, 1) if has_bwd else None,
        "roofline": roofline,
        "roofline_fwd": roof_fwd,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "overlap": "copies on their own streams, two device buffer sets",
                "passes_ms_per_step": [round(x, 4) for x in e2e_runs],
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_next_rows:
        result["next_rows"] = next_rows(args.seed)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, has_bwd, args.cpu_seconds)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def _time_ms(torch, fn, warm=3, reps=10):
    """Mean device time of fn() over `reps` back-to-back calls (CUDA events on
    the current stream), after `warm` untimed calls."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def next_rows(seed):
    """The widened rows, each timed on its own page's workload (synthetic
    inputs of that shape), outside the headline step's timed region:
      - Nystrom forward, bound by HBM: algorithmic bytes are Q twice (landmark
        pooling, output pass), K, V and O once;
      - Stieltjes forward, bound by the tensor cores: steps + 2 QK^T sweeps and
        one P.V per tile pair;
      - the packed variable-length forward and backward on a ragged causal GQA
        batch;
      - the deterministic backward, bound by the tensor cores (7 MMAs per tile
        pair counted as the 2.5x-forward convention's 5)."""
    import torch

    from flash_exact_attention_gb300 import binding
    from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

    hbm, hbm_src = _measured_hbm()
    peak_burst, _, peak_src = _measured_peaks()
    rows = {}

    def dev_inputs(B, Hq, Hkv, N, D, with_do=False):
        x = make_inputs(B, Hq, Hkv, N, D, seed, with_do=with_do)
        return {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}

    # Nystrom: the page's high batch x head shape and its long-context shape.
    for name, (B, H, N, D, m) in (("nystrom_b4_h16_n131072_d128_m64", (4, 16, 131072, 128, 64)),
                                  ("nystrom_b1_h4_n2097152_d64_m32", (1, 4, 2097152, 64, 32))):
        g = torch.Generator(device="cuda").manual_seed(seed)
        q, k, v = (torch.randn(B, H, N, D, device="cuda", generator=g).to(torch.bfloat16)
                   for _ in range(3))
        ms = _time_ms(torch, lambda: binding.nystrom_attn(q, k, v, num_landmarks=m,
                                                          newton_iters=6, kappa=5.0))
        st = binding.attn_device_status()
        if st:
            raise binding.AttnError(st, name)
        nbytes = 5 * B * H * N * D * 2
        gbs = nbytes / ms / 1e6
        rows[name] = {
            "workload": "Nystrom forward B=%d H=%d N=%d D=%d m=%d, 6 Newton-Schulz steps, "
                        "kappa 5 (iid N(0,1) bf16)" % (B, H, N, D, m),
            "metric": "forward latency", "value": round(ms, 4), "unit": "ms",
            "higher_is_better": False, "launches": 6,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4),
                         "traffic": _recorded_traffic("nystrom_call", name,
                                                      _kernel_source_hash(NYS_SOURCES)),
                         "algorithmic_bytes": nbytes,
                         "peak_source": "%s copy bandwidth" % hbm_src,
                         "timed_as": "whole attn_nystrom_fwd call (memset + 6 kernels)"}}
        del q, k, v
        torch.cuda.empty_cache()

    # Stieltjes attention, order 4, the page's three Newton steps.
    B, H, N, D = 2, 16, 8192, 128
    t = dev_inputs(B, H, H, N, D)
    ms = _time_ms(torch, lambda: binding.stieltjes_attn(t["q"], t["k"], t["v"], order=4,
                                                        newton_steps=3))
    st = binding.attn_device_status()
    if st:
        raise binding.AttnError(st, "stieltjes")
    att = 4.0 * B * H * N * N * D / ms / 1e9
    tensor = att / 2 * (3 + 2 + 1)
    rows["stieltjes_b2_h16_n8192_d128_q4"] = {
        "workload": "Stieltjes forward B=2 H=16 N=8192 D=128, order 4, 3 Newton steps",
        "metric": "attention TFLOPS (4 B H N^2 D per call)", "value": round(att, 1),
        "unit": "TFLOPS", "higher_is_better": True, "ms": round(ms, 4), "launches": 1,
        "roofline": {"bound": "tensor", "achieved": round(tensor, 1), "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": round(tensor / peak_burst, 4), "traffic": None,
                     "algorithmic_flops_per_launch": 2.0 * B * H * N * N * D * 6,
                     "peak_source": "%s bf16 burst" % peak_src}}

    # Ragged batch, packed without padding: causal GQA (Hq 16, Hkv 4, D 128),
    # 32 sequences of seeded lengths 1..8192 (about 130 k tokens).
    import numpy as np
    Hq, Hkv, D = 16, 4, 128
    lens = np.random.default_rng(seed).integers(1, 8193, size=32)
    total, ms_max = int(lens.sum()), int(lens.max())
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(total, Hq, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(total, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(total, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    ms = _time_ms(torch, lambda: binding.flash_attn_varlen(q, k, v, cu, ms_max, causal=True))
    st = binding.attn_device_status()
    if st:
        raise binding.AttnError(st, "varlen forward")
    flops = sum(4.0 * Hq * float(n) * float(n) * D / 2 for n in lens)
    tf = flops / ms / 1e9
    rows["varlen_causal_gqa_32seq_d128"] = {
        "workload": "packed ragged batch, causal GQA Hq=16 Hkv=4 D=128, 32 sequences of "
                    "seeded lengths 1..8192 (%d tokens, longest %d)" % (total, ms_max),
        "metric": "forward TFLOPS (sum over sequences of 2 Hq n^2 D)", "value": round(tf, 1),
        "unit": "TFLOPS", "higher_is_better": True, "ms": round(ms, 4), "launches": 1,
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4), "traffic": None,
                     "peak_source": "%s bf16 burst" % peak_src}}
    o, lse = binding.flash_attn_varlen(q, k, v, cu, ms_max, causal=True)
    do = torch.randn(total, Hq, D, device="cuda", generator=g).to(torch.bfloat16)
    ms = _time_ms(torch, lambda: binding.flash_attn_varlen_bwd(q, k, v, o, lse, do, cu, ms_max,
                                                               causal=True))
    st = binding.attn_device_status()
    if st:
        raise binding.AttnError(st, "varlen backward")
    tf = 2.5 * flops / ms / 1e9
    rows["varlen_bwd_causal_gqa_32seq_d128"] = {
        "workload": "backward of the same packed ragged batch (%d tokens)" % total,
        "metric": "backward TFLOPS (2.5x the forward's FLOPs)", "value": round(tf, 1),
        "unit": "TFLOPS", "higher_is_better": True, "ms": round(ms, 4),
        "launches": 3, "timed_as": "whole attn_bwd_varlen call (memset + 3 kernels)",
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4), "traffic": None,
                     "peak_source": "%s bf16 burst" % peak_src}}
    del q, k, v, cu, o, lse, do
    torch.cuda.empty_cache()

    # Deterministic backward on the headline shape.
    t = dev_inputs(B, H, H, N, D, with_do=True)
    o, lse = binding.flash_attn(t["q"], t["k"], t["v"])
    ms = _time_ms(torch, lambda: binding.flash_attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"],
                                                        deterministic=True))
    st = binding.attn_device_status()
    if st:
        raise binding.AttnError(st, "deterministic backward")
    tf = 2.5 * 4.0 * B * H * N * N * D / ms / 1e9
    rows["bwd_deterministic_b2_h16_n8192_d128"] = {
        "workload": "deterministic backward B=2 H=16 N=8192 D=128 non-causal",
        "metric": "backward TFLOPS (2.5x forward FLOPs)", "value": round(tf, 1),
        "unit": "TFLOPS", "higher_is_better": True, "ms": round(ms, 4), "launches": 3,
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4), "traffic": None,
                     "peak_source": "%s bf16 burst" % peak_src}}
    del t, o, lse
    torch.cuda.empty_cache()
    return rows


# Kernels the backward launches per call, and whether a step includes it.
BWD_LAUNCHES = 3
STEP_INCLUDES_BWD = True


def cpu_baseline(workload, with_bwd, budget_s):
    """The fp64 oracle, as it stands, on a bounded sample of the same workload."""
    import numpy as np

    import oracle
    from flash_exact_attention_gb300.synth import bf16_bits_to_f32, make_inputs, scale_for

    B, Hq, Hkv, N, D, causal, _ = WORKLOADS[workload]
    scale = scale_for(D)
    x = make_inputs(B, Hq, Hkv, N, D, seed=0, with_do=with_bwd)
    q, k, v = (bf16_bits_to_f32(x[n]) for n in ("q", "k", "v"))
    rng = np.random.default_rng(1)
    flops = 0.0
    t0 = time.perf_counter()
    rows_done = 0
    # forward on random rows in batches until the time budget is spent
    fwd_budget = budget_s / (3.5 if with_bwd else 1.0)
    while time.perf_counter() - t0 < fwd_budget:
        rows = rng.integers(0, B * Hq * N, size=max(64, oracle.num_threads() * 16))
        oracle.fwd_rows(q, k, v, causal, scale, rows)
        i = rows % N
        keys = (i + 1) if causal else np.full_like(i, N)
        flops += float(np.sum(4.0 * keys * D))
        rows_done += rows.size
    t_fwd = time.perf_counter() - t0
    sample = "forward of %d random rows" % rows_done
    t_bwd = 0.0
    if with_bwd:
        # backward of the first (batch, kv-head) group of the same workload
        t1 = time.perf_counter()
        sl = slice(0, Hq // Hkv)
        qq = q[:1, sl]
        kk = k[:1, :1]
        vv = v[:1, :1]
        dd = bf16_bits_to_f32(x["do"])[:1, sl]
        oracle.bwd(qq, kk, vv, dd, causal, scale)
        t_bwd = time.perf_counter() - t1
        flops += 2.5 * fwd_flops(1, Hq // Hkv, N, D, causal)
        sample += " + backward of one (batch, kv-head) group (%d query heads)" % (Hq // Hkv)
    secs = t_fwd + t_bwd
    return {"value": round(flops / secs / 1e12, 6), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle", "sample": sample,
            "seconds": round(secs, 2), "host_cpus": os.cpu_count()}


def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    has_bwd = STEP_INCLUDES_BWD
    B, Hq, Hkv, N, D, causal, desc = WORKLOADS[args.workload]
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        cpu_baseline(args.workload, has_bwd, 0.2)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(args.workload, has_bwd, args.cpu_seconds / max(1, args.steps)))
    wall = time.perf_counter() - t0
    value = statistics.median(v["value"] for v in vals)
    cb = dict(vals[-1])
    cb["value"] = value
    result = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * wall / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic iid N(0,1) bf16 from numpy seed 0",
        "config": {"workload": desc, "name": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv,
                   "N": N, "D": D, "causal": causal,
                   "step": "fwd+bwd" if has_bwd else "fwd",
                   "note": "the fp64 CPU oracle on a bounded sample of the workload per step"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(result), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-clock budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the widened rows (Nystrom, Stieltjes, varlen, deterministic "
                         "backward)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
