"""Benchmark of the gated delta-rule prefill and decode step on one GB300 per rank.

One JSON line on rank 0.  ``value`` is the prefill throughput (tokens/s =
B * S / time, summed over ranks) on the B=4, Hk=16, Hv=32, S=4096, Dk=Dv=128
bf16 workload with its inputs resident in HBM; the decode step (B=64, Hk=16,
Hv=32, Dk=Dv=128, 128 MiB fp32 state) is measured in the same run and
reported under ``decode`` in GB/s of algorithmic traffic.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own copy of the workload (independent
sequences, no collective): weak scaling.  ``--impl reference`` times the fp64
CPU oracle on the same workload instead (all sequences per step when the run fits about three
minutes, else a measured subset; the step time is measured, never extrapolated).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "GDN prefill tokens/s + tensor-pipe %; decode-step state GB/s vs HBM peak"
PREFILL = workloads.PREFILL
DECODE = workloads.DECODE_STEP
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.md")
KERNEL_SOURCES = {
    "gdn_prefill_tc_kernel": "gated_delta_rule_20_gb300/csrc/prefill_tc.cu",
    # the same kernel on the wide-GQA workload (its own traffic row)
    "gdn_prefill_tc_kernel_wide_gqa": "gated_delta_rule_20_gb300/csrc/prefill_tc.cu",
    "gdn_decode_stream_kernel": "gated_delta_rule_20_gb300/csrc/decode.cu",
    "conv1d_prefill_vec8_kernel": "gated_delta_rule_20_gb300/csrc/conv1d.cu",
    "conv1d_decode_k4_kernel": "gated_delta_rule_20_gb300/csrc/conv1d.cu",
    "gdn_decode_gated_stream_kernel": "gated_delta_rule_20_gb300/csrc/decode_gated.cu",
    "inproj_gemm_kernel": "gated_delta_rule_20_gb300/csrc/block.cu",
    "rmsnorm_gated_d128_kernel": "gated_delta_rule_20_gb300/csrc/rmsnorm_gated.cu",
    # the two kernels of one decode-block call; the sha covers both files, in this order
    "decode_block": ("gated_delta_rule_20_gb300/csrc/block.cu", "gated_delta_rule_20_gb300/csrc/decode_gated.cu"),
}


# ------------------------------------------------------------------ algorithmic accounting
def prefill_bytes(w) -> int:
    """Bytes the method must move once: q, k per key head; v, out per value
    head; g_log and beta; the fp32 state in (when supplied) and out."""
    e = 2 if w.dtype == "bf16" else 4
    qk = 2 * w.B * w.Hk * w.S * w.Dk * e
    v_out = 2 * w.B * w.Hv * w.S * w.Dv * e
    gb = 2 * w.B * w.Hv * w.S * 4
    st = (2 if w.state_std > 0 else 1) * w.B * w.Hv * w.Dk * w.Dv * 4
    return qk + v_out + gb + st


def prefill_flops(w, C=64) -> float:
    """Algorithmic flops at chunk C with causal triangles counted at half:
    per value-head token 6 Dk Dv + C (3 Dk + 2 Dv) + C^2 / 3."""
    per = 6 * w.Dk * w.Dv + C * (3 * w.Dk + 2 * w.Dv) + C * C / 3.0
    return per * w.B * w.Hv * w.S


def conv1d_bytes(w) -> int:
    """Algorithmic bytes of one conv1d call: x in, out, the fp32 weights, and the
    conv_state (written by the prefill; read and written by the decode step)."""
    esz = 2 if w.dtype == "bf16" else 4
    act = w.B * w.C * w.T * esz
    state = w.B * w.C * w.K * esz
    return 2 * act + w.C * w.K * 4 + state * (2 if w.kind == "decode" else 1)


def gated_bytes(w) -> int:
    """Algorithmic bytes of one gated decode step: the fp32 state in and out, the
    q|k|v row, z and out, a and b, and the per-head parameters."""
    esz = 2 if w.dtype == "bf16" else 4
    state = 2 * w.B * w.Hv * w.Dk * w.Dv * 4
    act = w.B * (2 * w.Hk * w.Dk + w.Hv * w.Dv) * esz + 2 * w.B * w.Hv * w.Dv * esz + 2 * w.B * w.Hv * esz
    return state + act + 2 * w.Hv * 4 + w.Dv * 4


def block_bytes(w) -> int:
    """Algorithmic bytes of one decode-block call: the four bf16 in_proj weights, the
    hidden row, the conv window and the fp32 state (each in and out), the conv
    weights, the per-head parameters and the output."""
    vd = w.Hv * w.Dv
    weights = w.H * (w.C + vd + 2 * w.Hv) * 2
    return (weights + w.B * w.H * 2 + 2 * w.B * w.C * w.K * 2 + 2 * w.B * w.Hv * w.Dk * w.Dv * 4 +
            w.C * w.K * 4 + 2 * w.Hv * 4 + w.Dv * 4 + w.B * vd * 2)


def norm_bytes(w) -> int:
    """Algorithmic bytes of the RMSNormGated pass over a prefill's output: the output
    read and rewritten, z read, and norm_weight."""
    e = 2 if w.dtype == "bf16" else 4
    return 3 * w.B * w.Hv * w.S * w.Dv * e + w.Dv * 4


def decode_bytes(w) -> int:
    e = 2 if w.dtype == "bf16" else 4
    return (2 * w.B * w.Hv * w.Dk * w.Dv * 4 + 2 * w.B * w.Hk * w.Dk * e + 2 * w.B * w.Hv * w.Dv * e
            + 2 * w.B * w.Hv * 4)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def code_sha(paths) -> str:
    """sha256[:16] of the sources' code with comments and blank lines removed, so that a
    comment edit does not invalidate a recorded capture but any code change does."""
    import hashlib
    import re
    text = b"".join(open(os.path.join(ROOT, f), "rb").read() for f in paths).decode()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.split("\n") if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current code of the kernel (else None)."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    srcs = KERNEL_SOURCES[kernel]
    sha = code_sha((srcs,) if isinstance(srcs, str) else srcs)
    for line in open(PROFILE_TRAFFIC):
        parts = line.strip().strip("|").split("|")
        parts = [p.strip() for p in parts]
        if len(parts) >= 3 and parts[0] == kernel and parts[2] == sha:
            try:
                return int(parts[1])
            except ValueError:
                return None
    return None


# ------------------------------------------------------------------ ranks
def rank_workload(w, rank: int):
    """Each rank runs its own copy of the workload with its own seed: the
    sequences are independent, so ranks never exchange data (weak scaling)."""
    return w.with_(seed=w.seed + 1000 * rank)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank time over all ranks (the only cross-rank operation
    besides barriers)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 20 ms; `summary` keeps those taken between
    `mark_start()` and `mark_end()` (the timed region)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "gdn_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = getattr(self, "t_start", 0.0) - 0.05
        t1 = getattr(self, "t_end", 1e30) + 0.05
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if ts is not None and not (t0 <= ts <= t1):
                continue
            try:
                sm.append(float(p[2]))
                mx.append(float(p[3]))
            except ValueError:
                continue
            for n, val in zip(names, p[6:10]):
                if val.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample(w, n_seq: int, seed: int = 0):
    """Oracle inputs for the first n_seq (batch, value-head) sequences of the workload."""
    import torch
    x = workloads.make_inputs(w)
    G = w.Hv // w.Hk
    heads = [(i // w.Hv, i % w.Hv) for i in range(n_seq)]
    pick = lambda t, kv: torch.stack([t[b, (h // G) if kv else h] for b, h in heads]).unsqueeze(1)
    return dict(q=pick(x["q"], True).double().numpy(), k=pick(x["k"], True).double().numpy(),
                v=pick(x["v"], False).double().numpy(), g=pick(x["g_log"], False).double().numpy(),
                beta=pick(x["beta"], False).double().numpy(),
                state=None if x["state"] is None else pick(x["state"], False).double().numpy(),
                scale=x["scale"])


def time_oracle(w, n_seq: int, sample=None):
    import oracle
    s = sample if sample is not None else oracle_sample(w, n_seq)
    t0 = time.perf_counter()
    oracle.recurrence(s["q"], s["k"], s["v"], s["g"], s["beta"], s["scale"], s["state"])
    dt = time.perf_counter() - t0
    full_time = dt * (w.B * w.Hv) / n_seq       # the whole workload at this rate
    return dict(seconds=dt, tokens_per_s=w.B * w.S / full_time, cores=oracle.max_threads())


# ------------------------------------------------------------------ our implementation
def sustained(torch, stream, calls, n_steps, nbytes, peak):
    """Back-to-back launches cycling through ``calls`` (one per input set, each set holding its
    own state, so that three sets are larger than L2 and no step finds its state in L2); one
    event pair around the whole loop.  The steady-state rate of a serving loop: launch latency
    overlaps the previous step, and no L2 flush runs (nor leaves dirty lines) in between."""
    for i in range(len(calls)):
        calls[i]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n_steps):
        calls[i % len(calls)]()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "value": gbs, "unit": "GB/s", "frac": gbs / peak, "steps": n_steps, "input_sets": len(calls),
            "method": "back-to-back launches over %d input sets, each with its own state (> L2 together)" % len(calls)}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import gated_delta_rule_20_gb300 as gdn

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---------------- prefill, inputs resident in HBM
    w = rank_workload(PREFILL, rank)
    x = workloads.make_inputs(w, device=dev)
    state = x["state"].clone()
    out = torch.empty((w.B, w.Hv, w.S, w.Dv), dtype=w.torch_dtype, device=dev)

    def prefill_step():
        gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], state, out, stream=stream)

    for _ in range(max(args.warmup, 3)):
        prefill_step()
    torch.cuda.synchronize()
    if gdn.device_status(local_rank) != 0:
        raise RuntimeError("prefill kernel reported a wait timeout")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        for i in range(args.steps):
            ev[i][0].record(stream)
            prefill_step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        barrier()
    clocks = clk.summary()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    ms_per_step = total_ms / args.steps
    ms_per_step = max_over_ranks(ms_per_step, world, dev)
    value = weak_scaling_value(w.B * w.S, world, ms_per_step)
    avg_launch_s = statistics.mean(launch_ms) * 1e-3
    pbytes = prefill_bytes(w)
    pflops = prefill_flops(w)
    roof = {"bound": "hbm", "achieved": pbytes / avg_launch_s / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": pbytes / avg_launch_s / 1e9 / peaks["hbm"], "traffic": recorded_traffic("gdn_prefill_tc_kernel"),
            "kernel": "gdn_prefill_tc_kernel", "algorithmic_bytes_per_launch": pbytes,
            "peak_source": peaks["source"] + " hbm_gbs",
            "tensor": {"achieved_tflops": pflops / avg_launch_s / 1e12, "peak": peaks["bf16"],
                       "peak_source": peaks["source"] + " bf16_tflops (burst: each launch is timed on its own)",
                       "frac": pflops / avg_launch_s / 1e12 / peaks["bf16"],
                       "frac_of_sustained": pflops / avg_launch_s / 1e12 / peaks["bf16_sustained"],
                       "algorithmic_flops_per_launch": pflops}}

    # ---------------- the gated prefill (the prefill, then RMSNormGated on its output), inputs > L2
    gz = workloads.make_gate_inputs(w, device=dev)
    gstate = x["state"].clone()
    gout = torch.empty_like(out)

    def gated_prefill_step():
        gdn.prefill_gated(x["q"], x["k"], x["v"], x["g_log"], x["beta"], gz["z"], gz["norm_weight"], x["scale"],
                          gstate, gout, stream=stream)

    for _ in range(max(args.warmup, 3)):
        gated_prefill_step()
    torch.cuda.synchronize()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(min(args.steps, 50))]
    for a_, b_ in gev:
        a_.record(stream)
        gated_prefill_step()
        b_.record(stream)
    torch.cuda.synchronize()
    gpms = statistics.median([a_.elapsed_time(b_) for a_, b_ in gev])
    nbytes = norm_bytes(w)
    prefill_gated = {"workload": w.name, "ms": gpms, "tokens_per_s": w.B * w.S / (gpms * 1e-3) * world,
                     "kernels": 2, "norm_pass_ms": gpms - statistics.median(launch_ms),
                     "norm_pass_roofline": {"bound": "hbm", "algorithmic_bytes_per_launch": nbytes,
                                            "achieved": nbytes / ((gpms - statistics.median(launch_ms)) * 1e-3) / 1e9,
                                            "peak": peaks["hbm"], "unit": "GB/s",
                                            "traffic": recorded_traffic("rmsnorm_gated_d128_kernel"),
                                            "kernel": "rmsnorm_gated_d128_kernel",
                                            "note": "norm pass time = gated-prefill median minus prefill median"}}
    prefill_gated["norm_pass_roofline"]["frac"] = prefill_gated["norm_pass_roofline"]["achieved"] / peaks["hbm"]
    del gz, gstate, gout

    # ---------------- decode step, L2 flushed between launches
    wd = rank_workload(DECODE, rank)
    xd = workloads.make_inputs(wd, device=dev)
    dstate = xd["state"].clone()
    dout = torch.empty((wd.B, wd.Hv, 1, wd.Dv), dtype=wd.torch_dtype, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def decode_step():
        gdn.decode_step(xd["q"], xd["k"], xd["v"], xd["g_log"], xd["beta"], xd["scale"], dstate, dout,
                        stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        decode_step()
    torch.cuda.synchronize()
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        dev_ev[i][0].record(stream)
        decode_step()
        dev_ev[i][1].record(stream)
    torch.cuda.synchronize()
    dms = statistics.median([a.elapsed_time(b) for a, b in dev_ev])
    dbytes = decode_bytes(wd)
    decode = {"value": dbytes / (dms * 1e-3) / 1e9 * world, "unit": "GB/s", "ms": dms,
              "workload": wd.name, "l2": "flushed (256 MiB write) before every launch",
              "roofline": {"bound": "hbm", "achieved": dbytes / (dms * 1e-3) / 1e9, "peak": peaks["hbm"],
                           "unit": "GB/s", "frac": dbytes / (dms * 1e-3) / 1e9 / peaks["hbm"],
                           "traffic": recorded_traffic("gdn_decode_stream_kernel"), "kernel": "gdn_decode_stream_kernel",
                           "algorithmic_bytes_per_launch": dbytes}}
    sets = [dict(xd, state=xd["state"].clone()) for _ in range(3)]
    decode["sustained"] = sustained(
        torch, stream, [lambda st=st_["state"]: gdn.decode_step(xd["q"], xd["k"], xd["v"], xd["g_log"], xd["beta"],
                                                                  xd["scale"], st, dout, stream=stream) for st_ in sets],
        max(30, min(args.steps, 300)), dbytes, peaks["hbm"])
    del xd, dstate, dout, sets

    roof["tensor_frac"] = roof["tensor"]["frac"]
    roof["decode_gbs"] = decode["roofline"]["achieved"]
    roof["decode_frac"] = decode["roofline"]["frac"]
    roof["decode_sustained_frac"] = decode["sustained"]["frac"]

    # ---------------- conv1d in front of the recurrence: prefill (input > L2) and decode (L2 flushed)
    conv = {}
    for wc in (workloads.CONV_PREFILL, workloads.CONV_DECODE):
        wc = wc.with_(seed=wc.seed + 100 * rank)
        xc = workloads.make_conv_inputs(wc, device=dev)
        cout = torch.empty_like(xc["x"])
        cst = xc["state"] if wc.kind == "decode" else torch.empty((wc.B, wc.C, wc.K), dtype=xc["x"].dtype,
                                                                   device=dev)
        if wc.kind == "prefill":
            call = lambda: gdn.conv1d_prefill(xc["x"], xc["weight"], out=cout, conv_state=cst, stream=stream)
        else:
            call = lambda: gdn.conv1d_decode(xc["x"], xc["weight"], cst, out=cout, stream=stream)
        for _ in range(max(args.warmup, 3)):
            if wc.kind == "decode":
                flush.zero_()
            call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            if wc.kind == "decode":
                flush.zero_()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        cms = statistics.median([a.elapsed_time(b) for a, b in ev])
        cb = conv1d_bytes(wc)
        kname = "conv1d_prefill_vec8_kernel" if wc.kind == "prefill" else "conv1d_decode_k4_kernel"
        conv[wc.kind] = {
            "workload": wc.name, "ms": cms, "tokens_per_s": wc.B * wc.T / (cms * 1e-3) * world,
            "l2": "input larger than L2" if wc.kind == "prefill" else "flushed (256 MiB write) before every launch",
            "roofline": {"bound": "hbm", "achieved": cb / (cms * 1e-3) / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": cb / (cms * 1e-3) / 1e9 / peaks["hbm"], "traffic": recorded_traffic(kname),
                         "kernel": kname, "algorithmic_bytes_per_launch": cb}}
        del xc, cout, cst

    # ---------------- gated decode step (prologue + recurrence + RMSNormGated), L2 flushed
    wg = workloads.GATED_DECODE.with_(seed=workloads.GATED_DECODE.seed + 100 * rank)
    xg = workloads.make_gated_inputs(wg, device=dev)
    gout = torch.empty((wg.B, wg.Hv * wg.Dv), dtype=wg.torch_dtype, device=dev)

    def gated_step():
        gdn.decode_gated(xg["qkv"], xg["z"], xg["a"], xg["b"], xg["A_log"], xg["dt_bias"], xg["norm_weight"],
                         xg["scale"], xg["state"], wg.Hk, wg.Hv, wg.Dk, wg.Dv, out=gout, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        gated_step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        gated_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    gms = statistics.median([a.elapsed_time(b) for a, b in ev])
    gb = gated_bytes(wg)
    gated = {"workload": wg.name, "ms": gms, "value": gb / (gms * 1e-3) / 1e9 * world, "unit": "GB/s",
             "l2": "flushed (256 MiB write) before every launch",
             "roofline": {"bound": "hbm", "achieved": gb / (gms * 1e-3) / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                          "frac": gb / (gms * 1e-3) / 1e9 / peaks["hbm"],
                          "traffic": recorded_traffic("gdn_decode_gated_stream_kernel"), "kernel": "gdn_decode_gated_stream_kernel",
                          "algorithmic_bytes_per_launch": gb}}
    gsets = [xg["state"].clone() for _ in range(3)]
    gated["sustained"] = sustained(
        torch, stream, [lambda st=st_: gdn.decode_gated(xg["qkv"], xg["z"], xg["a"], xg["b"], xg["A_log"], xg["dt_bias"],
                                                         xg["norm_weight"], xg["scale"], st, wg.Hk, wg.Hv, wg.Dk, wg.Dv,
                                                         out=gout, stream=stream) for st_ in gsets],
        max(30, min(args.steps, 300)), gb, peaks["hbm"])
    del xg, gout, gsets

    # ---------------- the decode block (in_proj GEMM with the conv window shift, then the gated step
    #                  with the conv output), L2 flushed
    wb = workloads.DECODE_BLOCK.with_(seed=workloads.DECODE_BLOCK.seed + 100 * rank)
    xb = workloads.make_block_inputs(wb, device=dev)
    bws = torch.empty(gdn.decode_block_workspace_bytes(wb.B, wb.H, wb.Hk, wb.Hv, wb.Dk, wb.Dv, wb.K),
                      dtype=torch.uint8, device=dev)
    bout = torch.empty((wb.B, 1, wb.Hv * wb.Dv), dtype=torch.bfloat16, device=dev)

    def block_step():
        gdn.decode_block(xb["hidden"], xb["W_qkv"], xb["W_z"], xb["W_a"], xb["W_b"], xb["conv_weight"],
                         xb["conv_state"], xb["A_log"], xb["dt_bias"], xb["norm_weight"], xb["state"], wb.Hk, wb.Hv,
                         wb.Dk, wb.Dv, out=bout, workspace=bws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        block_step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        block_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    bms = statistics.median([a.elapsed_time(b) for a, b in ev])
    bb = block_bytes(wb)
    block = {"workload": wb.name, "ms": bms, "tokens_per_s": wb.B / (bms * 1e-3) * world, "kernels": 2,
             "l2": "flushed (256 MiB write) before every call",
             "roofline": {"bound": "hbm", "achieved": bb / (bms * 1e-3) / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                          "frac": bb / (bms * 1e-3) / 1e9 / peaks["hbm"], "traffic": recorded_traffic("decode_block"),
                          "kernel": "inproj_gemm_kernel + gdn_decode_gated_stream_kernel",
                          "algorithmic_bytes_per_call": bb}}
    bsets = [workloads.make_block_inputs(wb.with_(seed=wb.seed + 1 + i), device=dev) for i in range(3)]
    block["sustained"] = sustained(
        torch, stream, [lambda t=t: gdn.decode_block(t["hidden"], t["W_qkv"], t["W_z"], t["W_a"], t["W_b"],
                                                     t["conv_weight"], t["conv_state"], t["A_log"], t["dt_bias"],
                                                     t["norm_weight"], t["state"], wb.Hk, wb.Hv, wb.Dk, wb.Dv,
                                                     out=bout, workspace=bws, stream=stream) for t in bsets],
        max(30, min(args.steps, 300)), bb, peaks["hbm"])
    block["sustained"]["method"] = "back-to-back calls over 3 input sets, each with its own weights and states"
    del xb, bws, bout, flush, bsets

    # ---------------- long sequences (B=1, Hv=32, S=32768, zero start): the default form, which splits
    #                  each sequence into segments over more SMs, against one pass (GDN_SINGLE_PASS)
    wl = rank_workload(workloads.LONG_PREFILL, rank)
    xl = workloads.make_inputs(wl, device=dev)
    lout = torch.empty((wl.B, wl.Hv, wl.S, wl.Dv), dtype=wl.torch_dtype, device=dev)
    lbytes, lflops = prefill_bytes(wl), prefill_flops(wl)
    # the split's scratch is the caller's (gdn_prefill_ws): the timed region allocates nothing
    lws_bytes = gdn.prefill_workspace_bytes(wl.B, wl.Hk, wl.Hv, wl.S, wl.Dk, wl.Dv)
    lws = torch.empty(max(lws_bytes, 16), dtype=torch.uint8, device=dev)

    def long_leg(single_pass):
        def step():
            gdn.prefill(xl["q"], xl["k"], xl["v"], xl["g_log"], xl["beta"], xl["scale"], None, lout,
                        single_pass=single_pass, stream=stream, workspace=lws)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        evl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(3, min(args.steps, 20)))]
        for a, b in evl:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.median([a.elapsed_time(b) for a, b in evl])
        return {"ms": ms, "tokens_per_s": wl.B * wl.S / (ms * 1e-3) * world,
                "hbm_frac": lbytes / (ms * 1e-3) / 1e9 / peaks["hbm"],
                "tensor_frac": lflops / (ms * 1e-3) / 1e12 / peaks["bf16"],
                "tensor_frac_of_sustained": lflops / (ms * 1e-3) / 1e12 / peaks["bf16_sustained"]}

    long_prefill = {"workload": wl.name, "split": long_leg(False), "single_pass": long_leg(True),
                    "algorithmic_bytes": lbytes, "algorithmic_flops": lflops,
                    "workspace_bytes": lws_bytes,
                    "segment_starts": gdn.prefill_segment_starts(wl.B, wl.Hk, wl.Hv, wl.S),
                    "note": "split: one launch of segment 0 and, per later segment, a zero-start and an "
                            "identity-start run (several CTA waves); a combine step; a tensor-core "
                            "correction of the later segments' outputs (plus an identity fill and a "
                            "memset); scratch in a caller workspace allocated before timing; inputs larger "
                            "than L2"}
    del xl, lout, lws

    # ---------------- wide-GQA batched prefill (B=16, Hk=8, Hv=32, S=2048: 512 sequences, 4 value heads
    #                  per key head), supplied state aliased in and out, inputs larger than L2
    wq = rank_workload(workloads.WIDE_GQA_PREFILL, rank)
    xq = workloads.make_inputs(wq, device=dev)
    qstate = xq["state"].clone()
    qout = torch.empty((wq.B, wq.Hv, wq.S, wq.Dv), dtype=wq.torch_dtype, device=dev)
    qbytes, qflops = prefill_bytes(wq), prefill_flops(wq)

    def gqa_step():
        gdn.prefill(xq["q"], xq["k"], xq["v"], xq["g_log"], xq["beta"], xq["scale"], qstate, qout, stream=stream)

    for _ in range(3):
        gqa_step()
    torch.cuda.synchronize()
    evq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(3, min(args.steps, 50)))]
    for a_, b_ in evq:
        a_.record(stream)
        gqa_step()
        b_.record(stream)
    torch.cuda.synchronize()
    qms = statistics.median([a_.elapsed_time(b_) for a_, b_ in evq])
    wide_gqa = {"workload": wq.name, "ms": qms, "tokens_per_s": wq.B * wq.S / (qms * 1e-3) * world,
                "algorithmic_bytes": qbytes, "algorithmic_flops": qflops,
                "hbm_frac": qbytes / (qms * 1e-3) / 1e9 / peaks["hbm"],
                "tensor_frac": qflops / (qms * 1e-3) / 1e12 / peaks["bf16"],
                "tensor_frac_of_sustained": qflops / (qms * 1e-3) / 1e12 / peaks["bf16_sustained"],
                "traffic": recorded_traffic("gdn_prefill_tc_kernel_wide_gqa"),
                "note": "q and k of a key head are read by its 4 value heads' CTAs; the algorithmic bytes "
                        "count them once per key head"}
    del xq, qstate, qout
    if gdn.device_status(local_rank) != 0:
        raise RuntimeError("a kernel reported a wait timeout")

    # ---------------- end to end through the public API from pinned host buffers
    # Every step copies its inputs and initial state from pinned host memory, runs gdn_prefill
    # and copies out and the final state back.  The copies of one step overlap the kernel and the
    # copies of its neighbours (three streams, device buffers double-buffered), as a serving loop
    # would run them; every byte of every step still crosses the link inside the timed region.
    xh = {k: (v.to("cpu").pin_memory() if hasattr(v, "to") and v is not None else v) for k, v in x.items()}
    st_h = xh["state"].clone().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    st_back = torch.empty(st_h.shape, dtype=torch.float32).pin_memory()
    bufs = [dict(q=torch.empty_like(x["q"]), k=torch.empty_like(x["k"]), v=torch.empty_like(x["v"]),
                 g=torch.empty_like(x["g_log"]), b=torch.empty_like(x["beta"]), st=torch.empty_like(state),
                 out=torch.empty_like(out)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (xh["q"], xh["k"], xh["v"], xh["g_log"], xh["beta"], st_h))
    d2h = out_h.numel() * out_h.element_size() + st_back.numel() * 4
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    d2h_done = [None, None]

    def e2e_step(i):
        bf = bufs[i & 1]
        with torch.cuda.stream(s_in):
            if d2h_done[i & 1] is not None:  # step i - 2 has read this buffer's out and state back
                s_in.wait_event(d2h_done[i & 1])
            for key, h_ in (("q", xh["q"]), ("k", xh["k"]), ("v", xh["v"]), ("g", xh["g_log"]), ("b", xh["beta"]),
                            ("st", st_h)):
                bf[key].copy_(h_, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        stream.wait_event(in_done)
        gdn.prefill(bf["q"], bf["k"], bf["v"], bf["g"], bf["b"], x["scale"], bf["st"], bf["out"], stream=stream)
        k_done = torch.cuda.Event()
        k_done.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(k_done)
            out_h.copy_(bf["out"], non_blocking=True)
            st_back.copy_(bf["st"], non_blocking=True)
            d2h_done[i & 1] = torch.cuda.Event()
            d2h_done[i & 1].record(s_out)

    for i in range(max(args.warmup, 3)):
        e2e_step(i)
    torch.cuda.synchronize()
    d2h_done[0] = d2h_done[1] = None
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 30))
    torch.cuda.synchronize()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(d2h_done[(e2e_steps - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e = {"value": weak_scaling_value(w.B * w.S, world, e2e_ms), "unit": "tokens/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "overlap": "copies of neighbouring steps overlap the kernel (3 streams, double-buffered device inputs)"}
    if gdn.device_status(local_rank) != 0:
        raise RuntimeError("a kernel reported a wait timeout")

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hk": w.Hk, "Hv": w.Hv, "S": w.S, "Dk": w.Dk, "Dv": w.Dv,
                   "parallelism": "independent sequences per rank" if world > 1 else "single gpu",
                   "l2": "inputs larger than L2 (%.0f MB per step)" % (pbytes / 1e6)},
        "roofline": roof, "prefill_gated": prefill_gated, "decode": decode, "decode_gated": gated, "decode_block": block, "conv1d": conv, "long_prefill": long_prefill, "wide_gqa_prefill": wide_gqa,
        "e2e": e2e, "clocks": clocks,
        "gpu_launches": args.steps * gdn.kernels_per_call(),
        "launch_ms": {"median": statistics.median(launch_ms), "min": min(launch_ms), "max": max(launch_ms)},
    }
    if rank == 0 and world == 1:
        n_seq = min(args.oracle_sequences, w.B * w.Hv)
        r = time_oracle(w, n_seq)
        result["cpu_baseline"] = {"value": r["tokens_per_s"], "unit": "tokens/s", "cores": r["cores"],
                                  "kind": "oracle",
                                  "sample": "%d of %d (batch, value-head) sequences, all %d tokens each, "
                                            "%.1f s wall%s" % (
                                                n_seq, w.B * w.Hv, w.S, r["seconds"],
                                                "" if n_seq == w.B * w.Hv else "; scaled to the whole workload")}
    return result


def run_reference(args):
    """The fp64 CPU oracle timed on the prefill workload, on every host core (OpenMP over the
    (batch, value-head) sequences).  Each step runs the oracle over all 128 sequences (about 0.7 s
    on 16 cores) unless --steps and --warmup would then take more than about three minutes, in
    which case each step runs the first n sequences, n sized to fit.  ms_per_step is the measured
    time of one step (nothing is extrapolated); the value is the tokens of the sequences a step
    runs over that time."""
    w = PREFILL
    total = w.B * w.Hv
    probe = oracle_sample(w, min(8, total))
    r = time_oracle(w, min(8, total), probe)
    per_seq = r["seconds"] / min(8, total)
    budget = 180.0 / (args.steps + args.warmup)
    n_seq = int(max(1, min(total, args.reference_sequences or total, budget / max(per_seq, 1e-9))))
    sample = oracle_sample(w, n_seq)
    for _ in range(args.warmup):
        time_oracle(w, n_seq, sample)
    times = []
    cores = 1
    for _ in range(args.steps):
        r = time_oracle(w, n_seq, sample)
        times.append(r["seconds"])
        cores = r["cores"]
    sec = statistics.mean(times)
    # the metric's tokens are the workload's B * S; a step over n_seq of the B * Hv sequences
    # covers that fraction of them
    value = w.B * w.S * (n_seq / total) / sec
    desc = ("%d of %d (batch, value-head) sequences x %d tokens per step, measured (not scaled)"
            % (n_seq, total, w.S))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hk": w.Hk, "Hv": w.Hv, "S": w.S, "Dk": w.Dk, "Dv": w.Dv,
                   "sequences_per_step": n_seq, "parallelism": "OpenMP over sequences on the host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--oracle-sequences", type=int, default=128)
    ap.add_argument("--reference-sequences", type=int, default=0,
                    help="sequences per reference step (0: all, or as many as fit about three minutes)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
