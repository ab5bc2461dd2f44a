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
# Sources of each kernel family: a recorded DRAM figure holds only while their
# hash is unchanged.
FAMILY_SOURCES = {
    "fwd_kernel": FWD_SOURCES + ["fwd_varlen_d128.cu", "fwd_varlen_d64.cu"],
    "bwd_kernel": BWD_SOURCES + ["bwd_varlen_d128.cu", "bwd_varlen_d64.cu", "bwd_det_d128.cu",
                                 "bwd_det_d64.cu"],
    "bwd_dq_kernel": ["bwd_dq_kernel.cuh", "ptx.cuh", "bwd_launch.cuh", "bwd_det_d128.cu",
                      "bwd_det_d64.cu"],
    "stj_kernel": ["stj_kernel.cuh", "ptx.cuh", "stj_d128.cu", "stj_d64.cu"],
    "nystrom_call": NYS_SOURCES,
}
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "dram_traffic.json")
# Kernel instantiations that only one of the widened rows launches (template
# arguments as ncu prints them, spaces removed, booleans as 0/1): their DRAM
# figures are recorded under that row's name whatever --workload says.
NEXT_ROW_KERNELS = {
    "stj_kernel<128,0,4>": "stieltjes_b2_h16_n8192_d128_q4",
    "fwd_kernel<128,1,0,1,0,0>": "varlen_causal_gqa_32seq_d128",
    "bwd_kernel<128,1,0,1,1>": "varlen_bwd_causal_gqa_32seq_d128",
    "bwd_kernel<128,0,0,0,0>": "bwd_deterministic_b2_h16_n8192_d128",
    "bwd_dq_kernel<128,0,0>": "bwd_deterministic_b2_h16_n8192_d128",
}


def _kernel_source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flash_exact_attention_gb300", "csrc")
    for n in sorted(set(names)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _recorded_traffic(family, workload, kernel=None):
    """DRAM bytes per launch of a kernel family on a workload, from
    profiles/dram_traffic.json, if recorded on the current sources (else None).
    `kernel` narrows the match to one instantiation ("fwd_kernel<128,...>")."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    src_hash = _kernel_source_hash(FAMILY_SOURCES[family])
    with open(TRAFFIC_JSON) as f:
        rows = json.load(f).get("rows", [])
    for r in rows:
        if (r.get("family") == family and r.get("workload") == workload
                and r.get("source_hash") == src_hash
                and (kernel is None or r.get("kernel") == kernel)):
            return float(r["dram_bytes_per_launch"])
    return None


def _traffic_or_why(family, workload, second_family=None):
    """{"traffic": bytes} from the recorded captures (the sum of both kernels
    when the call has two), or {"traffic": None, "traffic_note": why}."""
    t = _recorded_traffic(family, workload)
    if t is not None and second_family is not None:
        t2 = _recorded_traffic(second_family, workload)
        t = None if t2 is None else t + t2
    if t is None:
        return {"traffic": None,
                "traffic_note": "no ncu DRAM capture of this call on the current sources"}
    return {"traffic": t}


def _ncu_kernel_key(name):
    """'void fwd_kernel<128, 0, 0, 0, 0, 0>(...)' (ncu's form; also with an
    attn:: prefix, true/false or (bool)1/(bool)0) -> ('fwd_kernel',
    'fwd_kernel<128,0,0,0,0,0>')."""
    m = re.search(r"(?:void\s+)?(?:attn::)?(\w+)<([^>]*)>", name)
    if not m:
        m2 = re.search(r"(?:void\s+)?(?:attn::)?(\w+)", name)
        fam = m2.group(1) if m2 else name.strip()
        return fam, fam
    args = [a.strip() for a in m.group(2).split(",")]
    norm = {"true": "1", "false": "0", "(bool)1": "1", "(bool)0": "0"}
    args = [norm.get(a, a) for a in args]
    return m.group(1), "%s<%s>" % (m.group(1), ",".join(args))


def _read_ncu_csv(csv_path):
    """Launches of an ncu --csv capture: {launch id: {"name": kernel name,
    metric: value}} for the DRAM byte counters (bytes) and the duration (us)."""
    import csv
    launches = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        mname = row.get("Metric Name", "")
        if mname not in ("dram__bytes_read.sum", "dram__bytes_write.sum",
                         "gpu__time_duration.sum"):
            continue
        unit = (row.get("Metric Unit") or "").strip().lower()
        val = float(row["Metric Value"].replace(",", ""))
        scale = {"byte": 1, "b": 1, "kbyte": 1e3, "kb": 1e3, "mbyte": 1e6, "mb": 1e6,
                 "gbyte": 1e9, "gb": 1e9, "nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0,
                 "us": 1.0, "msecond": 1e3, "ms": 1e3, "second": 1e6, "s": 1e6}.get(unit, 1.0)
        d = launches.setdefault(row["ID"], {"name": row["Kernel Name"]})
        d[mname] = d.get(mname, 0.0) + val * scale
    return launches


def _launch_bytes(d):
    return d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"]


def _store_traffic_rows(recs):
    """Adds the records to the traffic file, each replacing the row of the same
    (family, kernel, workload)."""
    data = {"rows": []}
    if os.path.exists(TRAFFIC_JSON):
        with open(TRAFFIC_JSON) as f:
            data = json.load(f)
    rows = data.setdefault("rows", [])
    for rec in recs:
        rows[:] = [r for r in rows if not (r.get("family") == rec["family"]
                                           and r.get("kernel") == rec["kernel"]
                                           and r.get("workload") == rec["workload"])]
        rows.append(rec)
        print("recorded %s on %s: %.0f bytes per launch" % (rec["kernel"], rec["workload"],
                                                           rec["dram_bytes_per_launch"]))
    data["about"] = ("DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, "
                     "median over the captured launches) written by `python bench.py "
                     "--record-traffic <ncu csv> --workload <name>` (Nystrom: "
                     "`--record-nystrom-traffic`, one call summed over its six kernels); "
                     "bench.py uses a row only while the kernel family's source hash is "
                     "unchanged")
    rows.sort(key=lambda r: (r["workload"], r["family"], r["kernel"]))
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")


def record_traffic(csv_path, workload, command):
    """Reads an ncu --csv capture holding dram__bytes_read.sum and
    dram__bytes_write.sum per launch, and records the median bytes per launch of
    every kernel of the families above in profiles/dram_traffic.json, keyed by
    (family, instantiation, workload) with the current source hash."""
    per_kernel = {}
    for d in _read_ncu_csv(csv_path).values():
        fam, key = _ncu_kernel_key(d["name"])
        if fam not in FAMILY_SOURCES or "dram__bytes_read.sum" not in d:
            continue
        per_kernel.setdefault((fam, key), []).append(d)
    recs = []
    for (fam, key), ds in sorted(per_kernel.items()):
        rec = {"family": fam, "kernel": key, "workload": NEXT_ROW_KERNELS.get(key, workload),
               "source_hash": _kernel_source_hash(FAMILY_SOURCES[fam]),
               "dram_bytes_per_launch": round(statistics.median(_launch_bytes(x) for x in ds)),
               "launches": len(ds), "command": command}
        if all("gpu__time_duration.sum" in x for x in ds):
            rec["gpu_time_us_median_under_ncu"] = round(
                statistics.median(x["gpu__time_duration.sum"] for x in ds), 2)
        recs.append(rec)
    _store_traffic_rows(recs)


# The Nystrom call's six kernels; the three streaming passes' traffic grows
# with N, the other three (landmark algebra on m rows) do not.
NYS_STREAMING = ("nys_pool_kernel", "nys_kv_kernel", "nys_out_kernel")
NYS_KERNELS = NYS_STREAMING + ("nys_qt_kernel", "nys_merge_kernel", "nys_lmy_kernel")


def record_nystrom_traffic(csv_path, workload, scale, command):
    """DRAM bytes of one Nystrom call on `workload` from an ncu capture of the
    same call at N / scale (a full-size call holds too much device memory for a
    capture): per kernel the median bytes per launch, the streaming passes'
    times `scale`, summed over the six kernels.  Recorded as the row
    (nystrom_call, nystrom_call, workload)."""
    per = {}
    for d in _read_ncu_csv(csv_path).values():
        fam = _ncu_kernel_key(d["name"])[0]
        if fam in NYS_KERNELS and "dram__bytes_read.sum" in d:
            per.setdefault(fam, []).append(_launch_bytes(d))
    missing = [k for k in NYS_KERNELS if k not in per]
    if missing:
        raise SystemExit("capture lacks %s" % ", ".join(missing))
    parts = {k: statistics.median(v) * (scale if k in NYS_STREAMING else 1)
             for k, v in per.items()}
    _store_traffic_rows([{
        "family": "nystrom_call", "kernel": "nystrom_call", "workload": workload,
        "source_hash": _kernel_source_hash(FAMILY_SOURCES["nystrom_call"]),
        "dram_bytes_per_launch": round(sum(parts.values())), "launches": 1,
        "per_kernel_bytes": {k: round(v) for k, v in sorted(parts.items())},
        "captured_at": "N / %d, streaming passes scaled by %d" % (scale, scale),
        "command": command}])


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running.

    A reader thread stamps every sample with the host clock, so that one
    sampler can summarise several timed windows (``summary(t0, t1)``)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []  # (host time, sm MHz, max MHz, set of active reasons)
        self.thread = None

    def _read(self):
        import datetime
        for line in self.proc.stdout:
            c = [x.strip() for x in line.split(",")]
            if len(c) < 10:
                continue
            try:
                sm, smax = float(c[2]), float(c[3])
            except ValueError:
                continue
            # nvidia-smi's own local-time stamp (its output may reach the pipe
            # in late chunks); the arrival time if it does not parse
            try:
                when = datetime.datetime.strptime(c[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                when = time.time()
            active = {n for n, val in zip(self.REASONS, c[6:10]) if val.lower() == "active"}
            self.samples.append((when, sm, smax, active))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        # nvidia-smi's start-up briefly stalls the device; let it pass before timing.
        time.sleep(1.5)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in [t0, t1] (host time;
        the whole run when omitted).  Complete only after the sampler has exited."""
        sel = [x for x in self.samples
               if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        smax = sel[-1][2] if sel else (self.samples[-1][2] if self.samples else None)
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        reasons = set()
        for x in sel:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sel)}


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

    def roof(kernel, family, tflops, flops):
        h = _kernel_source_hash(FAMILY_SOURCES[family])
        return {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak_burst,
                "unit": "TFLOP/s", "frac": round(tflops / peak_burst, 4),
                "traffic": _recorded_traffic(family, args.workload), "kernel": kernel,
                "peak_source": peak_note, "frac_of_sustained": round(tflops / peak_sust, 4),
                "algorithmic_flops_per_launch": flops, "source_hash": h}

    roof_fwd = roof("fwd_kernel<%s>" % tag, "fwd_kernel", fwd_tflops, ff)
    if has_bwd:
        # The backward call (preprocess + main + postprocess, timed together) is
        # the dominant part of the step; its FLOPs are the main kernel's.
        roofline = roof("bwd_kernel<%s>" % tag, "bwd_kernel", bwd_tflops, 2.5 * ff)
        roofline["timed_as"] = "whole attn_bwd call (3 launches)"
    else:
        roofline = roof_fwd
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic iid N(0,1) bf16 from numpy seed %d (+rank)" % args.seed,
        "config": workload_config(args.workload, ws),
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
    if rank == 0 and not args.no_configs:
        result["configs"] = baseline_configs(args.seed, local)
    if rank == 0 and not args.no_next_rows:
        result["next_rows"] = next_rows(args.seed)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, has_bwd, args.cpu_reps)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# The five configurations the metric is quoted on (name, (B, Hq, Hkv, N, D,
# causal), what one step runs, description).  Configuration 4 is a sweep of
# three shapes of 16384 tokens per batch; configuration 2 has a ragged variant.
BASELINE_CONFIGS = (
    ("cfg1_b1_h2_n256_d64", (1, 2, 2, 256, 64, False), "fwd",
     "fwd, non-causal MHA, B=1 H=2 N=256 D=64"),
    ("cfg2_causal_b1_h16_n2048_d64", (1, 16, 16, 2048, 64, True), "fwd",
     "fwd, causal MHA, B=1 H=16 N=2048 D=64"),
    ("cfg2_causal_b1_h16_n2000_d64", (1, 16, 16, 2000, 64, True), "fwd",
     "fwd, causal MHA, B=1 H=16 N=2000 D=64 (ragged last tile)"),
    ("cfg3_causal_gqa_b1_hq8_hkv2_n4096_d128", (1, 8, 2, 4096, 128, True), "fwd",
     "fwd, causal GQA, B=1 Hq=8 Hkv=2 N=4096 D=128"),
    ("cfg4_b4_h16_n4096_d128", (4, 16, 16, 4096, 128, False), "fwd",
     "fwd, dense non-causal MHA, B=4 H=16 N=4096 D=128"),
    ("cfg4_b2_h16_n8192_d128", (2, 16, 16, 8192, 128, False), "fwd",
     "fwd, dense non-causal MHA, B=2 H=16 N=8192 D=128"),
    ("cfg4_b1_h16_n16384_d128", (1, 16, 16, 16384, 128, False), "fwd",
     "fwd, dense non-causal MHA, B=1 H=16 N=16384 D=128"),
    ("cfg5_causal_b1_h16_n4096_d64", (1, 16, 16, 4096, 64, True), "fwd+bwd",
     "fwd+bwd training step, causal MHA, B=1 H=16 N=4096 D=64"),
)


def min_fwd_bytes(B, Hq, Hkv, N, D):
    """Algorithmic forward traffic: Q, K, V read and O written once (16-bit),
    LSE written once (fp32)."""
    return 2 * (2 * B * Hq * N * D + 2 * B * Hkv * N * D) + 4 * B * Hq * N


def time_calls(torch, stream, fn, scrub, min_calls=20, min_seconds=0.3, warm=3):
    """Device time of fn() in ms, one pair of CUDA events per call on `stream`.
    With `scrub` (a buffer larger than L2) the buffer is written before every
    call, outside its events, so that each call starts from a cold L2.  Calls
    go on until at least `min_calls` and `min_seconds` of wall time (enough
    for the clock sampler to see the load).  Returns (times, host t0, host t1)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    times = []
    t0 = time.time()
    while len(times) < min_calls or time.time() - t0 < min_seconds:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min_calls)]
        for a, b in evs:
            if scrub is not None:
                scrub.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        times += [a.elapsed_time(b) for a, b in evs]
    return times, t0, time.time()


def baseline_configs(seed, local):
    """Every configuration of the metric, each on its own resident inputs,
    timed after the headline's timed region (CUDA events on the launch
    stream, L2 scrubbed before every call when the inputs fit in it)."""
    import torch

    from flash_exact_attention_gb300 import binding
    from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

    peak_burst, peak_sust, peak_src = _measured_peaks()
    hbm, hbm_src = _measured_hbm()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    scrub = torch.empty(256 * 2**20, dtype=torch.uint8, device="cuda")
    out, windows = {}, {}
    with ClockSampler(local) as clk:
        for name, (B, Hq, Hkv, N, D, causal), what, desc in BASELINE_CONFIGS:
            scale = scale_for(D)
            with_bwd = what == "fwd+bwd"
            x = make_inputs(B, Hq, Hkv, N, D, seed=seed, with_do=with_bwd)
            t = {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}
            o = torch.empty_like(t["q"])
            lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
            if with_bwd:
                dq, dk, dv = (torch.empty_like(t["q"]), torch.empty_like(t["k"]),
                              torch.empty_like(t["v"]))

            def fwd():
                st = binding.attn_fwd(t["q"], t["k"], t["v"], o, lse, B, Hq, Hkv, N, D, causal,
                                      scale, sh)
                if st:
                    raise binding.AttnError(st, "attn_fwd " + name)

            def bwd():
                st = binding.attn_bwd(t["q"], t["k"], t["v"], o, lse, B, Hq, Hkv, N, D, causal,
                                      scale, sh, t["do"], dq, dk, dv)
                if st:
                    raise binding.AttnError(st, "attn_bwd " + name)

            def step():
                fwd()
                bwd()

            in_bytes = sum(a.numel() * a.element_size() for a in t.values())
            cold = in_bytes < L2_BYTES
            ff = fwd_flops(B, Hq, N, D, causal)
            e = {"workload": desc, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "D": D,
                 "causal": causal, "step": what,
                 "l2": ("scrubbed: a 256 MiB buffer written before every call (inputs %.1f MiB "
                        "fit in the 129 MB L2)" % (in_bytes / 2**20)) if cold else
                       ("not scrubbed: inputs %.0f MiB exceed the 129 MB L2"
                        % (in_bytes / 2**20))}
            legs = (("step", step, 3.5 * ff), ("fwd", fwd, ff), ("bwd", bwd, 2.5 * ff)) \
                if with_bwd else (("fwd", fwd, ff),)
            w0 = None
            for leg, fn, flops in legs:
                times, a, b = time_calls(torch, stream, fn, scrub if cold else None)
                w0 = a if w0 is None else w0
                ms = statistics.fmean(times)
                e[leg + "_ms"] = round(ms, 5)
                e[leg + "_ms_median"] = round(statistics.median(times), 5)
                e[leg + "_tflops"] = round(flops / (ms * 1e-3) / 1e12, 2)
                e["calls"] = len(times)
            st = binding.attn_device_status(sh)
            if st:
                raise binding.AttnError(st, name)
            main = "step" if with_bwd else "fwd"
            tf = e[main + "_tflops"]
            e["tflops"] = tf
            e["pct_of_peak"] = round(100 * tf / peak_burst, 2)
            if name.startswith("cfg1"):
                # Four query tiles: a launch/latency-bound call.  Its figure is a
                # latency and the bandwidth of its minimal traffic, next to the
                # rate of back-to-back launches (warm L2, launches queued).
                nbytes = min_fwd_bytes(B, Hq, Hkv, N, D)
                ms = e["fwd_ms"]
                gbs = nbytes / (ms * 1e-3) / 1e9
                b2b, _, _ = time_calls(torch, stream, fwd, None)
                e["latency_us"] = round(1e3 * ms, 2)
                e["back_to_back_us_per_call"] = round(1e3 * statistics.fmean(b2b), 2)
                e["roofline"] = {
                    "bound": "latency", "achieved": round(gbs, 2), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 5), "algorithmic_bytes": nbytes,
                    "peak_source": "%s copy bandwidth" % hbm_src,
                    "note": "4 CTAs on 152 SMs: launch, first loads and the epilogue, not "
                            "bandwidth or tensor throughput, set the time"}
            else:
                e["roofline"] = {"bound": "tensor", "achieved": tf, "peak": peak_burst,
                                 "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4),
                                 "frac_of_sustained": round(tf / peak_sust, 4),
                                 "peak_source": "%s bf16 burst" % peak_src,
                                 "timed_as": "fwd+bwd step (attn_fwd + attn_bwd)" if with_bwd
                                 else "attn_fwd (one launch)"}
            windows[name] = (w0, time.time())
            out[name] = e
            del t, o, lse
            if with_bwd:
                del dq, dk, dv
            torch.cuda.empty_cache()
    for name, (a, b) in windows.items():  # every sample has been read by now
        out[name]["clocks"] = clk.summary(a, b)
    return out


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


NEXT_ROW_GROUPS = ("nystrom", "stieltjes", "varlen", "deterministic")


def next_rows(seed, only=NEXT_ROW_GROUPS):
    """The widened rows (the groups in `only`), each timed on its own page's workload (synthetic
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
    nys_shapes = (("nystrom_b4_h16_n131072_d128_m64", (4, 16, 131072, 128, 64)),
                  ("nystrom_b1_h4_n2097152_d64_m32", (1, 4, 2097152, 64, 32)))
    for name, (B, H, N, D, m) in (nys_shapes if "nystrom" in only else ()):
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
                         "traffic": _recorded_traffic("nystrom_call", name),
                         "algorithmic_bytes": nbytes,
                         "peak_source": "%s copy bandwidth" % hbm_src,
                         "timed_as": "whole attn_nystrom_fwd call (memset + 6 kernels)"}}
        del q, k, v
        torch.cuda.empty_cache()

    # Stieltjes attention, order 4, the page's three Newton steps.
    B, H, N, D = 2, 16, 8192, 128
    if "stieltjes" in only:
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
                         "unit": "TFLOP/s", "frac": round(tensor / peak_burst, 4),
                         **_traffic_or_why("stj_kernel", "stieltjes_b2_h16_n8192_d128_q4"),
                         "algorithmic_flops_per_launch": 2.0 * B * H * N * N * D * 6,
                         "peak_source": "%s bf16 burst" % peak_src}}

    if "varlen" in only:
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
                         "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4),
                         **_traffic_or_why("fwd_kernel", "varlen_causal_gqa_32seq_d128"),
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
                         "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4),
                         **_traffic_or_why("bwd_kernel", "varlen_bwd_causal_gqa_32seq_d128"),
                         "peak_source": "%s bf16 burst" % peak_src}}
        del q, k, v, cu, o, lse, do
        torch.cuda.empty_cache()

    if "deterministic" in only:
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
                         "unit": "TFLOP/s", "frac": round(tf / peak_burst, 4),
                         **_traffic_or_why("bwd_kernel", "bwd_deterministic_b2_h16_n8192_d128",
                                           "bwd_dq_kernel"),
                         "peak_source": "%s bf16 burst" % peak_src}}
        del t, o, lse
        torch.cuda.empty_cache()
    return rows


# Kernels the backward launches per call, and whether a step includes it.
BWD_LAUNCHES = 3
STEP_INCLUDES_BWD = True


# The oracle's fixed sample of a workload (the same in the CPU baseline of the
# native arm and in every step of the reference arm): the forward of
# ORACLE_FWD_ROWS query rows drawn with numpy seed 1, plus the backward of the
# first (batch, kv-head) group at full N.
ORACLE_FWD_ROWS = 2048


def oracle_sample(workload, with_bwd, inputs=None):
    """Runs the oracle's fixed sample once; returns (flops, seconds, description).
    FLOPs follow the metric's convention: 4*keys*D per forward row (keys = the
    row's allowed keys), 2.5x the forward of the group for its backward."""
    import numpy as np

    import oracle
    from flash_exact_attention_gb300.synth import bf16_bits_to_f32, make_inputs, scale_for

    B, Hq, Hkv, N, D, causal, _ = WORKLOADS[workload]
    scale = scale_for(D)
    if inputs is None:
        x = make_inputs(B, Hq, Hkv, N, D, seed=0, with_do=with_bwd)
        inputs = {n: bf16_bits_to_f32(a) for n, a in x.items()}
    q, k, v = inputs["q"], inputs["k"], inputs["v"]
    rows = np.random.default_rng(1).integers(0, B * Hq * N, size=ORACLE_FWD_ROWS)
    i = rows % N
    keys = (i + 1) if causal else np.full_like(i, N)
    flops = float(np.sum(4.0 * keys * D))
    t0 = time.perf_counter()
    oracle.fwd_rows(q, k, v, causal, scale, rows)
    desc = "forward of %d seeded rows" % ORACLE_FWD_ROWS
    G = Hq // Hkv
    if with_bwd:
        sl = slice(0, G)
        oracle.bwd(q[:1, sl], k[:1, :1], v[:1, :1], inputs["do"][:1, sl], causal, scale)
        flops += 2.5 * fwd_flops(1, G, N, D, causal)
        desc += " + backward of the (batch 0, kv-head 0) group (%d query head%s, N=%d)" % (
            G, "s" if G > 1 else "", N)
    return flops, time.perf_counter() - t0, desc


def _oracle_inputs(workload, with_bwd):
    from flash_exact_attention_gb300.synth import bf16_bits_to_f32, make_inputs
    B, Hq, Hkv, N, D, _, _ = WORKLOADS[workload]
    x = make_inputs(B, Hq, Hkv, N, D, seed=0, with_do=with_bwd)
    return {n: bf16_bits_to_f32(a) for n, a in x.items()}


def cpu_baseline(workload, with_bwd, reps=4):
    """The fp64 oracle, as it stands, on the host cores: its fixed sample of
    the workload, run `reps` times; the median rate."""
    import oracle
    inputs = _oracle_inputs(workload, with_bwd)
    runs = [oracle_sample(workload, with_bwd, inputs) for _ in range(reps)]
    rates = [f / sec / 1e12 for f, sec, _ in runs]
    return {"value": round(statistics.median(rates), 6), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": runs[0][2] + "; %d runs, median rate" % reps,
            "sample_flops": runs[0][0],
            "seconds": round(sum(sec for _, sec, _ in runs), 2), "host_cpus": os.cpu_count()}


def workload_config(workload, ws):
    """The `config` object of the JSON line (the same in both arms)."""
    B, Hq, Hkv, N, D, causal, desc = WORKLOADS[workload]
    x_bytes = 2 * (2 * B * Hq * N * D + 2 * B * Hkv * N * D)  # q, k, v, dO (16-bit)
    scrub = x_bytes < L2_BYTES
    return {"workload": desc, "name": workload, "B": B, "Hq": Hq, "Hkv": Hkv,
            "N": N, "D": D, "causal": causal,
            "step": "fwd+bwd" if STEP_INCLUDES_BWD else "fwd (backward not built)",
            "parallelism": "replicas" if ws == 1 else "dp%d (independent batches)" % ws,
            "l2": ("flushed: a 256 MiB buffer written before every timed step (inputs "
                   "%.0f MiB fit in the 129 MB L2; one pair of events per step)"
                   % (x_bytes / 2**20)) if scrub else
                  ("no flush: per-step inputs %.0f MiB exceed the 129 MB L2"
                   % (x_bytes / 2**20))}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle (there is no other
    implementation of the pages' method to install), each step its fixed
    sample of the workload, on the host cores."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    has_bwd = STEP_INCLUDES_BWD
    import oracle
    oracle.build()
    inputs = _oracle_inputs(args.workload, has_bwd)
    for _ in range(args.warmup):
        oracle_sample(args.workload, has_bwd, inputs)
    runs = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runs.append(oracle_sample(args.workload, has_bwd, inputs))
    wall = time.perf_counter() - t0
    flops = sum(f for f, _, _ in runs)
    secs = sum(sec for _, sec, _ in runs)
    value = round(flops / secs / 1e12, 6)
    cb = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
          "sample": runs[0][2] + " per step", "sample_flops": runs[0][0],
          "seconds": round(secs, 2), "host_cpus": os.cpu_count()}
    result = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * wall / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic iid N(0,1) bf16 from numpy seed %d (+rank)" % 0,
        "config": workload_config(args.workload, ws),
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
    ap.add_argument("--cpu-reps", type=int, default=4,
                    help="runs of the oracle's fixed sample in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other configurations of the metric")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the widened rows (Nystrom, Stieltjes, varlen, deterministic "
                         "backward)")
    ap.add_argument("--next-rows-only", metavar="GROUPS",
                    help="time only these widened rows (comma list of %s) and print them; "
                         "for profiling them alone" % ",".join(NEXT_ROW_GROUPS))
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="record the DRAM bytes per launch of an ncu --csv capture (metrics "
                         "dram__bytes_read.sum, dram__bytes_write.sum) taken on --workload "
                         "into profiles/dram_traffic.json, then exit")
    ap.add_argument("--record-nystrom-traffic", nargs=3, metavar=("NCU_CSV", "ROW", "SCALE"),
                    help="record one Nystrom call's DRAM bytes for the widened row ROW from "
                         "an ncu --csv capture of the same call at N / SCALE, then exit")
    ap.add_argument("--record-command", default="",
                    help="the ncu command line the capture came from (stored beside it)")
    ap.add_argument("--traffic-json", default=None,
                    help="file the records go to (default profiles/dram_traffic.json)")
    args = ap.parse_args()
    if args.record_traffic or args.record_nystrom_traffic:
        global TRAFFIC_JSON
        if args.traffic_json:
            TRAFFIC_JSON = args.traffic_json
        if args.record_traffic:
            record_traffic(args.record_traffic, args.workload, args.record_command)
        else:
            csv_path, row, scale = args.record_nystrom_traffic
            record_nystrom_traffic(csv_path, row, int(scale), args.record_command)
        return
    if args.next_rows_only:
        groups = tuple(g for g in args.next_rows_only.split(",") if g)
        bad = [g for g in groups if g not in NEXT_ROW_GROUPS]
        if bad:
            ap.error("unknown row groups: %s" % ",".join(bad))
        import torch
        torch.cuda.set_device(_dist_env()[2])
        print(json.dumps({"next_rows": next_rows(args.seed, groups)}), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
