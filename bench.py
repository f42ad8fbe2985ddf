"""Benchmark of the DSC hot path on B300.

One step = the whole hot path over one batch at C=6144, W=4:
  head-wise DSC forward + backward on the QKV placement
      (B=8, T=2048, C=6144, H=16 -> w [8,2048,384,4], bf16, residual), and
  low-rank fused DSC forward + backward on the same x shape
      (R=16, H=1, U [16, 24576], bf16, residual).
The metric is achieved HBM GB/s: the algorithmic (compulsory) bytes of the
four calls -- every tensor read or written once, halos and partial sums
excluded -- divided by the step time.  Inputs (0.45 GB and 0.40 GB per call)
are larger than the 126 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dsc|reference]

Under torchrun each rank runs the full workload on its own GPU (independent
replicas; no data-path collective), the timing is max over ranks, and the
value is the bytes of all ranks over that time.

--compare-static adds a second JSON line: per-call latency of the static
short convolution (w [C, W]) next to head-wise DSC at H=1 and H=16, same
shape, same GPU.

--sweep adds a line with per-shape throughput (GB/s, fraction of the
measured HBM peak, Mtokens/s) of the 27 all-linear placement shapes x both
parameterisations and the linear-RNN shape, forward and backward.

--impl reference times the fp64 CPU oracle on the host cores instead, each
step a bounded sample (the first 128 tokens of one sequence) of the same
workload; it prints the same JSON line with "impl": "reference".
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lm_local_sequence_causal_b300 import dsc, synthetic as syn  # noqa: E402

METRIC = "DSC fwd+bwd achieved HBM GB/s (% of B300 peak) and Mtokens/s at C=6144, W=4"
WORKLOAD = ("DSC at C=6144 W=4, B=8 T=2048 (16384 tokens), bf16, residual: head-wise "
            "H=16 fwd+bwd and low-rank R=16 H=1 fwd+bwd")
KERNEL_SOURCES = {
    "headwise_fwd": "lm_local_sequence_causal_b300/csrc/headwise_tma.cu",
    "headwise_bwd": "lm_local_sequence_causal_b300/csrc/headwise_tma.cu",
    "lowrank_fwd": "lm_local_sequence_causal_b300/csrc/lowrank_tc.cu",
    "lowrank_bwd": "lm_local_sequence_causal_b300/csrc/lowrank_tc.cu",
}
# What bounds each entry point as built: its roofline denominator.
KERNEL_BOUND = {"headwise_fwd": "hbm", "headwise_bwd": "hbm",
                "lowrank_fwd": "hbm", "lowrank_bwd": "hbm"}
# fp32 FMA peak of the CUDA cores: 148 SMs x 128 lanes x 2 flop x 2.032 GHz.
ALU_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12
FALLBACK_HBM_GBS = 6400.0
# GPU spin before the timed region's start event (about 2 ms at 2 GHz).
SPIN_CYCLES = 4_000_000


# ------------------------------------------------------------ byte model ----

def algorithmic(wl):
    """(fwd bytes, bwd bytes, fwd flops, bwd flops) of one call pair."""
    s = torch.empty((), dtype=wl.dtype).element_size()
    N, C, G, W, R = wl.tokens, wl.C, wl.G, wl.W, wl.R
    if wl.lowrank:
        fb = s * (2 * N * C + N * R + R * G * W)
        bb = s * (3 * N * C + 2 * N * R + 2 * R * G * W)
        ff = 2 * N * G * W * R + 2 * N * C * W
        bf = 6 * N * G * W * R + 3 * N * C * W
    else:
        fb = s * (2 * N * C + N * G * W)
        bb = s * (3 * N * C + 2 * N * G * W)
        ff = 2 * N * C * W
        bf = 4 * N * C * W
    return fb, bb, ff, bf


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(path):
    with open(os.path.join(ROOT, path), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def recorded_traffic(name):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(name)
    if not e or e.get("source_sha256_16") != source_hash(KERNEL_SOURCES[name]):
        return None
    return e.get("bytes_per_launch")


def entry_of_kernel(name):
    """The entry point a kernel of this library belongs to, from its ncu name."""
    m = re.search(r"hw_tma_kernel<\s*\d+,\s*\d+,\s*(\d)", name)
    if m:
        return "headwise_bwd" if m.group(1) == "1" else "headwise_fwd"
    if "lr_fwd_tc" in name:
        return "lowrank_fwd"
    if any(k in name for k in ("lr_u_image", "lr_bwd_tc", "lr_reduce_tc")):
        return "lowrank_bwd"
    return None


def record_traffic(csv_path, command, out_path=None):
    """Write the per-entry-point DRAM traffic record from an ncu launch list
    (`--metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum
    --csv`) of whole bench steps; bytes are per call (summed over the entry
    point's launches, divided by the number of calls captured)."""
    import csv
    with open(csv_path) as fh:
        lines = [l for l in fh if l.startswith('"')]
    launches = {}
    for r in csv.DictReader(lines):
        e = launches.setdefault(r["ID"], {"name": r["Kernel Name"]})
        e[r["Metric Name"]] = float(r["Metric Value"])
    sums, calls = {}, {}
    for e in launches.values():
        ent = entry_of_kernel(e["name"])
        if ent is None:
            continue
        s = sums.setdefault(ent, {"read": 0.0, "write": 0.0})
        s["read"] += e.get("dram__bytes_read.sum", 0.0)
        s["write"] += e.get("dram__bytes_write.sum", 0.0)
        main = ("hw_tma_kernel" in e["name"] or "lr_fwd_tc" in e["name"]
                or "lr_bwd_tc" in e["name"])
        calls[ent] = calls.get(ent, 0) + (1 if main else 0)
    out = {"_note": (
        "DRAM bytes (read + write) per call of each entry point at the QKV size "
        "(B=8 T=2048 C=6144 W=4 bf16), from one ncu pass over whole bench steps: "
        f"`{command}`, written by `python3 bench.py --record-traffic <that csv>`. "
        "Writes still dirty in L2 when a launch ends are counted in later launches. "
        "An entry is used only while the hash of its kernel source matches.")}
    for ent in ("headwise_fwd", "headwise_bwd", "lowrank_fwd", "lowrank_bwd"):
        if ent not in sums or not calls.get(ent):
            continue
        n = calls[ent]
        rd, wr = int(sums[ent]["read"] / n), int(sums[ent]["write"] / n)
        out[ent] = {"bytes_per_launch": rd + wr, "read": rd, "write": wr,
                    "source_sha256_16": source_hash(KERNEL_SOURCES[ent])}
        if ent == "lowrank_bwd":
            out[ent]["launches"] = "lr_u_image + lr_bwd_tc + lr_reduce_tc"
    p = out_path or os.path.join(ROOT, "profiles", "dram_traffic.json")
    with open(p, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    return out


# ------------------------------------------------------------ clocks --------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms from before
    the warm-up until after the timed region (the region itself can be as
    short as ten milliseconds); only samples taken between mark() and stop()
    are summarised."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device):
        import threading
        self.proc = None
        self.lines = []            # (host time, line)
        self.t_mark = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            gid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", gid],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.time()                       # wait for the first sample (at most 5 s)
        while not self.lines and time.time() - t0 < 5 and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def mark(self):
        """Start of the window that stop() summarises (before the warm-up)."""
        self.t_mark = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        n_end = len(self.lines)
        t0 = time.time()                       # one more sample after the timed region
        while len(self.lines) <= n_end and time.time() - t0 < 1 and self.proc.poll() is None:
            time.sleep(0.005)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        for t, line in self.lines:
            if self.t_mark is not None and t < self.t_mark:
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "warm-up and timed region, 20 ms interval"}


# ------------------------------------------------------------ the step ------

class Problem:
    """Device buffers for one step of the hot path."""

    def __init__(self, device, seed=0):
        self.hw = syn.qkv_headwise()
        self.lr = syn.qkv_lowrank()
        self.a = syn.make_inputs(self.hw, seed, device=device)
        self.b = syn.make_inputs(self.lr, seed + 1, device=device)
        a, b = self.a, self.b
        self.y_hw = torch.empty_like(a["x"])
        self.dx_hw = torch.empty_like(a["x"])
        self.dw_hw = torch.empty_like(a["w"])
        self.y_lr = torch.empty_like(b["x"])
        self.dx_lr = torch.empty_like(b["x"])
        self.dz_lr = torch.empty_like(b["z"])
        self.dU_lr = torch.empty_like(b["U"])
        self.ws = dsc.lowrank_workspace(b["x"], b["z"], self.lr.H, self.lr.W)

    def calls(self):
        """The four C calls of one step through the public binding (what a
        user writes); every call re-marshals its arguments."""
        a, b, hw, lr = self.a, self.b, self.hw, self.lr
        return [
            ("headwise_fwd", lambda: dsc.dsc_headwise_fwd(a["x"], a["w"], self.y_hw, hw.H, True)),
            ("headwise_bwd", lambda: dsc.dsc_headwise_bwd(a["x"], a["w"], a["dy"], self.dx_hw,
                                                          self.dw_hw, hw.H, True)),
            ("lowrank_fwd", lambda: dsc.dsc_lowrank_fwd(b["x"], b["z"], b["U"], self.y_lr,
                                                        lr.H, lr.W, True)),
            ("lowrank_bwd", lambda: dsc.dsc_lowrank_bwd(b["x"], b["z"], b["U"], b["dy"],
                                                        self.dx_lr, self.dz_lr, self.dU_lr,
                                                        self.ws, lr.H, lr.W, True)),
        ]

    def bound_calls(self, stream):
        """The same four C calls with their arguments marshalled once
        (dsc.bind), so that a timed loop spends its host time on the calls
        themselves and the GPU is never left waiting on Python."""
        a, b, hw, lr = self.a, self.b, self.hw, self.lr
        return [
            ("headwise_fwd", dsc.bind("dsc_headwise_fwd", a["x"], a["w"], self.y_hw, hw.H, True,
                                      stream)),
            ("headwise_bwd", dsc.bind("dsc_headwise_bwd", a["x"], a["w"], a["dy"], self.dx_hw,
                                      self.dw_hw, hw.H, True, stream)),
            ("lowrank_fwd", dsc.bind("dsc_lowrank_fwd", b["x"], b["z"], b["U"], self.y_lr,
                                     lr.H, lr.W, True, stream)),
            ("lowrank_bwd", dsc.bind("dsc_lowrank_bwd", b["x"], b["z"], b["U"], b["dy"],
                                     self.dx_lr, self.dz_lr, self.dU_lr, self.ws, lr.H, lr.W,
                                     True, stream)),
        ]

    # hw fwd, hw bwd, lr fwd, lr bwd (U image, main kernel, partial-sum reduction)
    LAUNCHES_PER_STEP = 6

    def bytes_flops(self):
        hf, hb, hff, hbf = algorithmic(self.hw)
        lf, lb, lff, lbf = algorithmic(self.lr)
        return ({"headwise_fwd": hf, "headwise_bwd": hb, "lowrank_fwd": lf, "lowrank_bwd": lb},
                {"headwise_fwd": hff, "headwise_bwd": hbf, "lowrank_fwd": lff,
                 "lowrank_bwd": lbf})

    def input_tensors(self):
        return [self.a["x"], self.a["w"], self.a["dy"], self.b["x"], self.b["z"], self.b["U"],
                self.b["dy"]]

    def output_tensors(self):
        return [self.y_hw, self.dx_hw, self.dw_hw, self.y_lr, self.dx_lr, self.dz_lr, self.dU_lr]


# ------------------------------------------------------------ distributed ---

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("gloo")


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(v, ws):
    if ws == 1:
        return v
    t = torch.tensor([float(v)], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle ----

def oracle_pass(sample_hw, sample_lr):
    """One fp64 oracle pass of the hot path over a sample; returns seconds."""
    return oracle_headwise(sample_hw) + oracle_lowrank(sample_lr)


def oracle_headwise(hw):
    """fp64 oracle forward + backward of the head-wise workload; seconds."""
    import oracle as orc
    t0 = time.perf_counter()
    orc.headwise_fwd(hw["x"], hw["w"], 16, True)
    orc.headwise_bwd(hw["x"], hw["w"], hw["dy"], 16, True)
    return time.perf_counter() - t0


def oracle_lowrank(lr):
    """fp64 oracle forward + backward of the low-rank workload; seconds."""
    import oracle as orc
    t0 = time.perf_counter()
    orc.lowrank_fwd(lr["x"], lr["z"], lr["U"], 1, 4, True)
    orc.lowrank_bwd(lr["x"], lr["z"], lr["U"], lr["dy"], 1, 4, True)
    return time.perf_counter() - t0


def sample_inputs(full, nseq, ntok):
    out = {}
    for k, v in full.items():
        out[k] = v.cpu() if k == "U" else v[:nseq, :ntok].contiguous().cpu()
    return out


def sample_bytes(nseq, ntok):
    hw = syn.qkv_headwise().with_(B=nseq, T=ntok)
    lr = syn.qkv_lowrank().with_(B=nseq, T=ntok)
    hf, hb, _, _ = algorithmic(hw)
    lf, lb, _, _ = algorithmic(lr)
    return hf + hb + lf + lb


def _leg(sec, nbytes, ntok):
    return {"seconds": round(sec, 3), "gbs": round(nbytes / sec / 1e9, 4),
            "mtok_per_s": round(ntok / sec / 1e6, 6)}


def cpu_baseline(prob):
    """The fp64 oracle on the host cores: the whole step (all 8 sequences of
    both workloads) on every thread, and one sequence of each workload on
    one thread; head-wise and low-rank legs timed separately."""
    import oracle as orc
    allc = orc.num_threads()
    hwb = sum(algorithmic(syn.qkv_headwise().with_(B=1))[:2])     # bytes per sequence
    lrb = sum(algorithmic(syn.qkv_lowrank().with_(B=1))[:2])
    T = 2048
    legs = {}
    s_hw, s_lr = sample_inputs(prob.a, 8, T), sample_inputs(prob.b, 8, T)
    th, tl = oracle_headwise(s_hw), oracle_lowrank(s_lr)
    legs["all_threads"] = {"threads": allc, "sample": "8 sequences (16384 tokens) per workload",
                           "headwise_C1": _leg(th, 8 * hwb, 8 * T),
                           "lowrank_C2": _leg(tl, 8 * lrb, 8 * T),
                           "step": _leg(th + tl, 8 * (hwb + lrb), 8 * T)}
    s_hw, s_lr = sample_inputs(prob.a, 1, T), sample_inputs(prob.b, 1, T)
    orc.set_num_threads(1)
    try:
        th1, tl1 = oracle_headwise(s_hw), oracle_lowrank(s_lr)
    finally:
        orc.set_num_threads(allc)
    legs["one_thread"] = {"threads": 1, "sample": "1 sequence (2048 tokens) per workload",
                          "headwise_C1": _leg(th1, hwb, T), "lowrank_C2": _leg(tl1, lrb, T),
                          "step": _leg(th1 + tl1, hwb + lrb, T)}
    step = legs["all_threads"]["step"]
    return {"value": step["gbs"], "unit": "GB/s", "cores": allc, "kind": "oracle",
            "sample": f"whole step (8 of 8 sequences, 16384 tokens, of both workloads, fwd+bwd, "
                      f"fp64) on {allc} threads: {step['seconds']} s; also one sequence of each "
                      f"workload on 1 thread",
            "seconds": step["seconds"], "mtok_per_s": step["mtok_per_s"], "legs": legs}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as orc
    hw = syn.qkv_headwise().with_(B=1, T=128)
    lr = syn.qkv_lowrank().with_(B=1, T=128)
    s_hw = syn.make_inputs(hw, 0)
    s_lr = syn.make_inputs(lr, 1)
    for _ in range(args.warmup):
        oracle_pass(s_hw, s_lr)
    tot = 0.0
    for _ in range(args.steps):
        tot += oracle_pass(s_hw, s_lr)
    sec = tot / args.steps
    nbytes = sample_bytes(1, 128)
    gbs = nbytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(),
        "cpu_baseline": {"kind": "oracle", "cores": orc.num_threads(),
                         "sample": "first 128 tokens of one sequence of both workloads, "
                                   "fwd+bwd, fp64 oracle on the host cores",
                         "value": round(gbs, 4)},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "mtok_per_s": round(128 / sec / 1e6, 6),
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict():
    return {"workload": WORKLOAD, "B": 8, "T": 2048, "C": 6144, "W": 4,
            "headwise_H": 16, "lowrank_R": 16, "lowrank_H": 1, "residual": True,
            "l2": "inputs larger than L2 (0.45 GB / 0.40 GB per call), no flush",
            "parallelism": "replicas (one full workload per GPU)"}


# ------------------------------------------------------------ main ----------

def run_dsc(args):
    ws, rank, local = dist_env()
    init_dist(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsc.load()
    prob = Problem(dev, seed=0)
    stream = torch.cuda.current_stream()
    calls = prob.bound_calls(stream)
    nbytes, nflops = prob.bytes_flops()
    step_bytes = sum(nbytes.values())

    # The clock sampler runs from before the warm-up to after the timed
    # region, and the timed region follows the warm-up with no idle gap.
    clocks = ClockSampler(dev)
    clocks.mark()
    for _ in range(args.warmup):
        for _, f in calls:
            f()
    # per-call events inside the timed region, on the launching stream;
    # created here so that the timed loop only records them
    ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)] for name, _ in calls}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    # A short GPU spin ahead of the start event lets the host enqueue the
    # first steps before the GPU reaches them, so the device-timed region
    # holds kernels back to back rather than the host's launch latency (the
    # host cost is reported separately, and the e2e line includes it).
    torch.cuda._sleep(SPIN_CYCLES)
    t_host = time.perf_counter()
    start.record(stream)
    for i in range(args.steps):
        for name, f in calls:
            e0, e1 = ev[name][i]
            e0.record(stream)
            f()
            e1.record(stream)
    end.record(stream)
    host_ms = (time.perf_counter() - t_host) * 1e3 / args.steps
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, ws)
    per_call_ms = {n: sum(a.elapsed_time(b) for a, b in v) / len(v) for n, v in ev.items()}

    # end to end: pinned host inputs -> device, the four calls, outputs -> host
    e2e = None
    if args.e2e_steps > 0:
        prob2 = Problem(dev, seed=0)          # the second buffer set of the pipeline
        e2e = run_e2e([prob, prob2], args.e2e_steps)
        del prob2
        torch.cuda.empty_cache()
    if e2e is not None:
        e2e_ms = max_over_ranks(e2e["ms_per_step"], ws)
        e2e["value"] = round(ws * step_bytes / (e2e_ms * 1e-3) / 1e9, 2)
        e2e["ms_per_step"] = round(e2e_ms, 3)

    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    value = ws * step_bytes / (ms * 1e-3) / 1e9
    dom = max(per_call_ms, key=per_call_ms.get)
    bound = KERNEL_BOUND[dom]
    if bound == "hbm":
        achieved = nbytes[dom] / (per_call_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
    else:
        achieved = nflops[dom] / (per_call_ms[dom] * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": round(achieved, 2),
                "peak": round(ALU_PEAK_TFLOPS, 2), "unit": "TFLOP/s",
                "frac": round(achieved / ALU_PEAK_TFLOPS, 4)}
    roof.update({"kernel": dom, "traffic": recorded_traffic(dom),
                 "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if bound == "hbm"
                 else "derived: 148 SMs x 128 fp32 lanes x 2 flop x 2.032 GHz"})
    kernels = {}
    for n in per_call_ms:
        t = per_call_ms[n] * 1e-3
        kernels[n] = {"ms": round(per_call_ms[n], 4), "gbs": round(nbytes[n] / t / 1e9, 1),
                      "frac_of_hbm_peak": round(nbytes[n] / t / 1e9 / peak, 4),
                      "tflops": round(nflops[n] / t / 1e12, 2), "bound": KERNEL_BOUND[n]}
    N = prob.hw.tokens
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(),
        "frac_of_hbm_peak": round(value / ws / peak, 4), "peak_gbs": peak,
        "mtok_per_s": {
            "headwise": round(N / ((per_call_ms["headwise_fwd"] + per_call_ms["headwise_bwd"])
                                   * 1e-3) / 1e6, 2),
            "lowrank": round(N / ((per_call_ms["lowrank_fwd"] + per_call_ms["lowrank_bwd"])
                                  * 1e-3) / 1e6, 2)},
        "kernels": kernels, "roofline": roof,
        "gpu_launches": Problem.LAUNCHES_PER_STEP * args.steps,
        "host_enqueue_ms_per_step": round(host_ms, 4),
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob)
    print(json.dumps(line), flush=True)
    if args.compare_static:
        print(json.dumps(run_compare_static(dev, min(args.steps, 100))), flush=True)
    if args.compare_decode:
        print(json.dumps(run_compare_decode(dev, min(args.steps, 100), measured_peaks()[0])),
              flush=True)
    if args.sweep:
        print(json.dumps(run_sweep(dev, args.sweep_calls)), flush=True)
    return 0


def run_compare_static(dev, steps):
    """Latency of the static short convolution (one filter per channel) next
    to the dynamic ones at the bench shape: the comparison the pages draw
    between DSC kernels and static short-conv kernels (their Figure 1), with
    both sides built here and run on the same GPU."""
    B, T, C, W = 8, 2048, 6144, 4
    dt = torch.bfloat16
    x = syn.draw((B, T, C), 1.0, 3, syn.SLOT_X, dt, dev)
    dy = syn.draw((B, T, C), 1.0, 3, syn.SLOT_DY, dt, dev)
    w = syn.static_filters(C, W, 0.5, 3, dt, dev)
    y, dx, dw = torch.empty_like(x), torch.empty_like(x), torch.empty_like(w)
    ws = torch.empty(max(dsc.dsc_static_bwd_workspace_size(B, T, C, W, dt), 16),
                     dtype=torch.uint8, device=dev)
    w1 = syn.draw((B, T, C, W), 0.5, 3, syn.SLOT_W, dt, dev)
    dw1 = torch.empty_like(w1)
    w16 = syn.draw((B, T, C // 16, W), 0.5, 4, syn.SLOT_W, dt, dev)
    dw16 = torch.empty_like(w16)
    cases = [
        ("static_fwd", lambda: dsc.dsc_static_fwd(x, w, y, True)),
        ("static_bwd", lambda: dsc.dsc_static_bwd(x, w, dy, dx, dw, ws, True)),
        ("headwise_H1_fwd", lambda: dsc.dsc_headwise_fwd(x, w1, y, 1, True)),
        ("headwise_H1_bwd", lambda: dsc.dsc_headwise_bwd(x, w1, dy, dx, dw1, 1, True)),
        ("headwise_H16_fwd", lambda: dsc.dsc_headwise_fwd(x, w16, y, 16, True)),
        ("headwise_H16_bwd", lambda: dsc.dsc_headwise_bwd(x, w16, dy, dx, dw16, 16, True)),
    ]
    stream = torch.cuda.current_stream()
    out = {}
    for name, f in cases:
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(steps):
            f()
        e.record(stream)
        torch.cuda.synchronize()
        out[name] = round(s.elapsed_time(e) / steps * 1e3, 2)
    return {"comparison": "static_vs_dynamic_short_conv", "unit": "us_per_call",
            "config": {"B": B, "T": T, "C": C, "W": W, "dtype": "bf16", "residual": True},
            "us": out}


def run_compare_decode(dev, steps, peak_gbs):
    """The decode step merged with its projection (one kernel,
    dsc_headwise_proj_decode) next to the unmerged pair (the projection as a
    cuBLAS matmul writing x, then dsc_headwise_decode), at the decode shape
    of the QKV placement: hidden D = 2048, C = 6144 (q, k, v), H = 16, W = 4,
    bf16, for B = 1, 4, 8, 16, 32, 64 and 256 sequences (and the low-rank step,
    R = 16, H = 1, for B = 1, 8 and 64).  Eight layers' inputs (eight Wp of
    25 MB: 201 MB, more than L2) are cycled, so each call reads its Wp from
    HBM as consecutive layers of a model do; the time per call is the event
    time of `steps` passes over the eight layers divided by the calls."""
    D, C, H, W, NL = 2048, 6144, 16, 4, 8
    dt = torch.bfloat16
    stream = torch.cuda.current_stream()
    res = {}
    for B in (1, 4, 8, 16, 32, 64, 256):
        layers = [syn.proj_decode_inputs(B, D, C, H, W, 0, dt, seed=10 + i, device=dev)
                  for i in range(NL)]
        x = torch.empty(B, C, dtype=dt, device=dev)
        y = torch.empty(B, C, dtype=dt, device=dev)
        fused = [dsc.bind("dsc_headwise_proj_decode", L["h"], L["Wp"], L["w"], L["state"], y, H,
                          True) for L in layers]
        steps_ = [dsc.bind("dsc_headwise_decode", x, L["w"], L["state"], y, H, True)
                  for L in layers]

        def run_fused():
            for f in fused:
                f()

        def run_unmerged():
            for L, f in zip(layers, steps_):
                torch.mm(L["h"], L["Wp"].t(), out=x)
                f()

        out = {}
        for name, f in (("merged", run_fused), ("unmerged", run_unmerged)):
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(SPIN_CYCLES)
            a.record(stream)
            for _ in range(steps):
                f()
            b.record(stream)
            torch.cuda.synchronize()
            out[name] = a.elapsed_time(b) / (steps * NL) * 1e3
        nbytes = 2 * (C * D + B * D + B * (C // H) * W + 2 * B * (W - 1) * C + B * C)
        gbs = nbytes / (out["merged"] * 1e-6) / 1e9
        res[str(B)] = {"merged_us": round(out["merged"], 2),
                       "unmerged_us": round(out["unmerged"], 2),
                       "speedup": round(out["unmerged"] / out["merged"], 3),
                       "merged_gbs": round(gbs, 1),
                       "merged_frac_of_hbm_peak": round(gbs / peak_gbs, 4),
                       "bytes_per_call": nbytes}
    # the low-rank step (R = 16, H = 1): taps z U formed in the kernel
    res_lr = {}
    R = 16
    for B in (1, 8, 64):
        layers = [syn.proj_decode_inputs(B, D, C, 1, W, R, dt, seed=40 + i, device=dev)
                  for i in range(NL)]
        x = torch.empty(B, C, dtype=dt, device=dev)
        y = torch.empty(B, C, dtype=dt, device=dev)
        fused = [dsc.bind("dsc_lowrank_proj_decode", L["h"], L["Wp"], L["z"], L["U"], L["state"],
                          y, 1, W, True) for L in layers]
        steps_ = [dsc.bind("dsc_lowrank_decode", x, L["z"], L["U"], L["state"], y, 1, W, True)
                  for L in layers]

        def run_fused_lr():
            for f in fused:
                f()

        def run_unmerged_lr():
            for L, f in zip(layers, steps_):
                torch.mm(L["h"], L["Wp"].t(), out=x)
                f()

        out = {}
        for name, f in (("merged", run_fused_lr), ("unmerged", run_unmerged_lr)):
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(SPIN_CYCLES)
            a.record(stream)
            for _ in range(steps):
                f()
            b.record(stream)
            torch.cuda.synchronize()
            out[name] = a.elapsed_time(b) / (steps * NL) * 1e3
        res_lr[str(B)] = {"merged_us": round(out["merged"], 2),
                          "unmerged_us": round(out["unmerged"], 2),
                          "speedup": round(out["unmerged"] / out["merged"], 3)}
    return {"comparison": "decode_step_merged_with_its_projection_vs_unmerged",
            "unit": "us_per_call", "kernel_launches_per_call": {"merged": 1, "unmerged": 2},
            "config": {"D": D, "C": C, "H": H, "W": W, "dtype": "bf16", "residual": True,
                       "layers_cycled": NL, "l2": "eight layers' weights (201 MB) cycled"},
            "peak_gbs": peak_gbs, "B": res,
            "lowrank": {"config": {"R": R, "H": 1}, "B": res_lr}}


def _time_calls(f, n, stream, flush):
    """Mean device time (ms) of n calls of f, each bracketed by its own event
    pair, with `flush` (a write larger than L2) between calls and outside the
    pairs; 3 warm-up calls first, and a GPU spin ahead of the first call keeps
    the host ahead of the GPU."""
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda._sleep(SPIN_CYCLES)
    for a, b in ev:
        flush()
        a.record(stream)
        f()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / n


def run_sweep(dev, n):
    """Throughput of every all-linear placement shape (C in {2048, 6144,
    5632} x T in {512, 2048, 8192} at 16384 tokens x W in {2, 3, 4}, head-wise
    H=16 and low-rank R=16) and of the linear-RNN shape (B=2, T=16384,
    C=4096, W=4; H=64 and R=16), forward and backward timed separately."""
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # 2x the L2

    def flush():
        scrub.fill_(1)

    rows = []
    wls = syn.all_linear_sweep() + [syn.linear_rnn_headwise(), syn.linear_rnn_lowrank()]
    for wl in wls:
        inp = syn.make_inputs(wl, 0, device=dev)
        x, dy = inp["x"], inp["dy"]
        y, dx = torch.empty_like(x), torch.empty_like(x)
        if wl.lowrank:
            z, U = inp["z"], inp["U"]
            dz, dU = torch.empty_like(z), torch.empty_like(U)
            ws = dsc.lowrank_workspace(x, z, wl.H, wl.W)
            fwd = dsc.bind("dsc_lowrank_fwd", x, z, U, y, wl.H, wl.W, wl.residual, stream)
            bwd = dsc.bind("dsc_lowrank_bwd", x, z, U, dy, dx, dz, dU, ws, wl.H, wl.W,
                           wl.residual, stream)
            path = dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R,
                                                     wl.dtype)
            path = {"fwd": "tcgen05" if path & 1 else "cuda_cores",
                    "bwd": "tcgen05" if path & 2 else "cuda_cores"}
        else:
            w = inp["w"]
            dw = torch.empty_like(w)
            fwd = dsc.bind("dsc_headwise_fwd", x, w, y, wl.H, wl.residual, stream)
            bwd = dsc.bind("dsc_headwise_bwd", x, w, dy, dx, dw, wl.H, wl.residual, stream)
            path = dsc.dsc_headwise_uses_tma(wl.B, wl.T, wl.C, wl.H, wl.W, wl.dtype)
            path = {"fwd": "tma" if path & 1 else "register_streaming",
                    "bwd": "tma" if path & 2 else "register_streaming"}
        fb, bb, _, _ = algorithmic(wl)
        tf, tb = _time_calls(fwd, n, stream, flush), _time_calls(bwd, n, stream, flush)
        rows.append({
            "name": wl.name, "B": wl.B, "T": wl.T, "C": wl.C, "W": wl.W, "H": wl.H,
            "R": wl.R, "path": path,
            "fwd_us": round(tf * 1e3, 1), "bwd_us": round(tb * 1e3, 1),
            "fwd_gbs": round(fb / tf / 1e6, 1), "bwd_gbs": round(bb / tb / 1e6, 1),
            "fwd_frac": round(fb / tf / 1e6 / peak, 4), "bwd_frac": round(bb / tb / 1e6 / peak, 4),
            "fwd_bwd_gbs": round((fb + bb) / (tf + tb) / 1e6, 1),
            "fwd_bwd_frac": round((fb + bb) / (tf + tb) / 1e6 / peak, 4),
            "mtok_per_s": round(wl.tokens / ((tf + tb) * 1e-3) / 1e6, 2)})
        del inp, x, dy, y, dx, fwd, bwd
        torch.cuda.empty_cache()
    return {"sweep": "all_linear_and_linear_rnn", "unit": "GB/s of algorithmic bytes",
            "peak_gbs": peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
            "calls_per_point": n, "dtype": "bf16", "residual": True, "data": "synthetic",
            "l2": "L2 flushed (256 MB write) before every timed call; each call timed by "
                  "its own event pair", "rows": rows}


def run_e2e(probs, steps):
    """The same metric through the public API with host buffers: every step
    copies all of its inputs from pinned host memory and reads every output
    back.  Consecutive steps are pipelined the way a training loop over
    host-resident data would run them: two device buffer sets (`probs`)
    alternate, the host->device copies of step i+1 run on one stream and the
    device->host copies of step i on another while the calls run on the
    current stream (the host link is full duplex), with events ordering
    every reuse of a buffer set."""
    h_in = [t.cpu().pin_memory() for t in probs[0].input_tensors()]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
             for t in probs[0].output_tensors()]
    ins = [p.input_tensors() for p in probs]
    outs = [p.output_tensors() for p in probs]
    calls = [p.calls() for p in probs]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in probs]
    ev_comp = [torch.cuda.Event() for _ in probs]
    ev_out = [torch.cuda.Event() for _ in probs]
    for e in ev_comp + ev_out:
        e.record(comp)
    bi = sum(t.numel() * t.element_size() for t in ins[0])
    bo = sum(t.numel() * t.element_size() for t in outs[0])

    def step(i):
        k = i % len(probs)
        s_in.wait_event(ev_comp[k])          # set k's inputs are free once its calls ended
        with torch.cuda.stream(s_in):
            for d, h in zip(ins[k], h_in):
                d.copy_(h, non_blocking=True)
        ev_in[k].record(s_in)
        comp.wait_event(ev_in[k])
        comp.wait_event(ev_out[k])           # set k's outputs have been read back
        for _, f in calls[k]:
            f()
        ev_comp[k].record(comp)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            for h, d in zip(h_out, outs[k]):
                h.copy_(d, non_blocking=True)
        ev_out[k].record(s_out)

    for i in range(len(probs)):
        step(i)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(comp)
    s_in.wait_event(s)
    s_out.wait_event(s)
    for i in range(steps):
        step(i)
    for ev in ev_out:
        comp.wait_event(ev)
    e.record(comp)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return {"value": None, "unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": ms, "steps": steps,
            "copies": "pinned host buffers; the input copies of step i+1 and the output copies "
                      "of step i overlap (two device buffer sets, one copy stream each way)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dsc", choices=["dsc", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compare-static", action="store_true",
                    help="also print a second line: static short conv vs DSC latency")
    ap.add_argument("--compare-static-only", action="store_true",
                    help="print only the static-vs-DSC latency line (single GPU)")
    ap.add_argument("--sweep", action="store_true",
                    help="also print a line with per-shape throughput of the all-linear "
                         "placement sweep and the linear-RNN shape")
    ap.add_argument("--sweep-only", action="store_true",
                    help="print only the sweep line (single GPU)")
    ap.add_argument("--sweep-calls", type=int, default=20)
    ap.add_argument("--compare-decode", action="store_true",
                    help="also print a line: the decode step merged with its projection "
                         "vs the unmerged pair")
    ap.add_argument("--compare-decode-only", action="store_true",
                    help="print only that line (single GPU)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="host only: write profiles/dram_traffic.json from an ncu launch list "
                         "of whole bench steps, then exit")
    ap.add_argument("--record-command", default="",
                    help="the ncu command that produced --record-traffic's CSV (for the note)")
    args = ap.parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.record_command), indent=1))
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.compare_decode_only:
        torch.cuda.set_device(0)
        dsc.load()
        print(json.dumps(run_compare_decode(torch.device("cuda", 0), min(args.steps, 100),
                                            measured_peaks()[0])), flush=True)
        return 0
    if args.compare_static_only:
        torch.cuda.set_device(0)
        dsc.load()
        print(json.dumps(run_compare_static(torch.device("cuda", 0), min(args.steps, 100))),
              flush=True)
        return 0
    if args.sweep_only:
        torch.cuda.set_device(0)
        dsc.load()
        print(json.dumps(run_sweep(torch.device("cuda", 0), args.sweep_calls)), flush=True)
        return 0
    return run_dsc(args)


if __name__ == "__main__":
    sys.exit(main())
