#!/usr/bin/env python
"""Benchmark of the H3 attention hot path on GB300.

One step = one pass of the whole path over one packed sequence (batch 1):
QK-RMSNorm + 3-axis RoPE of q and k written straight into the Ulysses
head-sharded layout (fused with seq->head), seq->head of v with degree P,
attention of each of the P head groups (one h3attn_forward call per group, as
each rank of a P-way group would issue it), head->seq of the output.

The default workload is the 480p-like packed sequence: 56 heads x 128,
49,920 video tokens (32 x 30 x 52) + 992 audio tokens padded to 51,200 keys
with a key-padding mask.  Inputs are seeded synthetic N(0,1) bf16 (no dataset,
no trained weights); each tensor is 734 MB, larger than L2, so no L2 flush is
needed between steps.

Output: ONE JSON line on rank 0.  `value` is attention TFLOP/s over the whole
job: 4 * S_v^2 * D * H per sequence (valid tokens only), summed over ranks,
divided by the max-over-ranks wall time of the timed steps.

--impl reference times the fp64 CPU oracle (the plain definition of the same
computation) on the host cores, on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own independent sequence (weak
scaling, no data-path collective); torch.distributed is used only for the
barrier and the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attention TFLOPS & tokens/s at 56 heads×128, 50k-262k tokens; % of bf16 peak")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HBM_SPEC_GBS = 7900.0            # HBM3e spec-sheet bandwidth, reported beside the measured copy figure
BF16_FLOP_PER_CLK_SM = 8192.0    # dense bf16 tcgen05 rate per SM per clock (M128 N128 K16 in 64 cycles)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attention_dram_traffic.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["h3attn", "reference"], default="h3attn")
    ap.add_argument("--workload", default="480p", choices=["c2", "16k", "480p", "1080p"])
    ap.add_argument("--P", type=int, default=2, help="Ulysses degree emulated inside one step")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-proj", action="store_true", help="skip timing the all-gather variant's fp8 projection")
    ap.add_argument("--graph", action="store_true", help="also time the step replayed as a CUDA graph (StepGraph)")
    ap.add_argument("--long-steps", type=int, default=3,
                    help="timed steps of the 1080p leg that follows a shorter headline workload (0: skip it)")
    ap.add_argument("--long-warmup", type=int, default=2)
    ap.add_argument("--no-chunks", action="store_true",
                    help="skip timing the step with head-chunked attention and overlapped output exchange")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--ulysses", choices=["a2a", "ag"], default=None,
                    help="time the Ulysses step ACROSS ranks instead (one sequence, S/N rows per rank, strong "
                         "scaling): a2a = all-to-all of q, k, v; ag = all-gather of the fp8 hidden state")
    return ap.parse_args()


def load_peaks(path=None):
    """Roofline denominators: the measured peaks file when present (flat or
    nested JSON with hbm_gbs / bf16_tflops / bf16_tflops_sustained), else the
    fallback figures.  Returns (peaks, "measured" | "fallback")."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            flat = {}

            def walk(x, prefix=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{prefix}{k}.")
                elif isinstance(x, (int, float)):
                    flat[prefix[:-1]] = float(x)
            walk(d)

            def pick(*names):
                for n in names:
                    for k, v in flat.items():
                        if k.split(".")[-1] == n:
                            return v
                return None
            hbm = pick("hbm_gbs", "hbm_GBps", "copy_gbs")
            b = pick("bf16_tflops", "bf16_tflops_burst")
            bs = pick("bf16_tflops_sustained")
            if hbm and b:
                return {"hbm_gbs": hbm, "bf16_tflops": b, "bf16_tflops_sustained": bs or b}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


ATTN_SOURCES = [os.path.join(ROOT, "dit_sequence_attention_gb300", "csrc", f)
                for f in ("attention.cu", "h3_device.cuh")]


def attention_fingerprint():
    """sha256 (first 16 hex digits) of the attention kernel's sources."""
    import hashlib
    h = hashlib.sha256()
    for path in ATTN_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, or None when that capture was taken on other kernel sources
    (the summary records the fingerprint of the sources it measured)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, None
    vals = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith(" "):
                key, val = line.split(":", 1)
                vals[key.strip()] = val.strip().split()[0] if val.strip() else ""
    fp = vals.get("attention_sources_sha256_16")
    try:
        traffic = float(vals["traffic_bytes_per_launch_480p_group28"])
    except (KeyError, ValueError):
        return None, None
    if fp != attention_fingerprint():
        return None, "committed capture is of other attention sources"
    return traffic, "profiles/attention_dram_traffic.txt (committed ncu capture of the same kernel sources)"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        return self.summarize(text)

    @staticmethod
    def summarize(text):
        """Median SM clock, median instantaneous board power and the throttle
        reasons seen in nvidia-smi's CSV output; None without a usable sample.
        (The plain power.draw field is a one-second average, which lags a
        timed region of about a second.)"""
        rows = list(csv.reader(io.StringIO(text)))
        if len(rows) < 2:
            return None
        hdr = [h.strip() for h in rows[0]]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows[1:]:
            if len(r) != len(hdr):
                continue
            rec = dict(zip(hdr, [x.strip() for x in r]))
            try:
                sm.append(float(rec[[h for h in hdr if h.startswith("clocks.current.sm") or h.startswith("clocks.sm")][0]].split()[0]))
                smax.append(float(rec[[h for h in hdr if h.startswith("clocks.max.sm")][0]].split()[0]))
            except Exception:
                continue
            try:
                power.append(float(rec[[h for h in hdr if h.startswith("power.draw")][0]].split()[0]))
            except Exception:
                pass
            for n in names:
                key = [h for h in hdr if h.startswith(f"clocks_event_reasons.{n}")]
                if key and rec[key[0]].lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
               "samples": len(sm)}
        if power:
            out["power_w"] = statistics.median(power)
        return out


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
        backend = "nccl" if args.impl == "h3attn" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (identity on one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the work every rank did over the slowest rank's time."""
    return flops_per_rank_step * steps * world / (max_ms * 1e-3) / 1e12


def cpu_oracle_sample(w, target_s, seed_offset=0):
    """Time the fp64 oracle on a bounded sample of workload `w`: QK-norm + RoPE of
    the sampled heads' keys and query rows, then attention of the sampled rows
    against every valid key.  Returns (flops_attention, seconds, description, threads)."""
    import numpy as np
    import oracle
    from dit_sequence_attention_gb300 import synth
    oracle.build()
    rng = np.random.default_rng(7 + seed_offset)
    pos = synth.packed_positions(w)
    wq, wk = synth.norm_weights(w.D)
    wq64, wk64 = wq.double().numpy(), wk.double().numpy()
    # one head's q/k/v (per-head draws keep host memory small; the oracle sees bf16-exact values)
    gen = lambda seed: synth.randn_bf16((w.S, 1, w.D), 1000 + seed + seed_offset, zero_rows_from=w.S_v)
    qh, kh, vh = (oracle.bf16_to_f64(gen(s)) for s in (1, 2, 3))

    def run(rows):
        t0 = time.perf_counter()
        kr = oracle.norm_rope(kh, wk64, pos, w.eps, *w.rope_split, w.theta)
        qr = oracle.norm_rope(qh[rows], wq64, pos[rows], w.eps, *w.rope_split, w.theta)
        oracle.attention(qr, kr, vh, kv_len=w.S_v)
        return time.perf_counter() - t0

    rows = np.sort(rng.choice(w.S, 16, replace=False))
    t_small = run(rows)
    n = int(min(w.S, max(16, 16 * target_s / max(t_small, 1e-3))))
    rows = np.sort(rng.choice(w.S, n, replace=False))
    dt = run(rows)
    flops = 4.0 * n * w.S_v * w.D
    desc = (f"1 head x {n} sampled query rows (QK-norm+RoPE of those rows and all {w.S} keys, "
            f"then attention over {w.S_v} valid keys) of the {w.name} workload")
    return flops, dt, desc, oracle.num_threads()


def run_reference(args, world, rank):
    """--impl reference: the fp64 CPU oracle on the host cores, rank 0 only."""
    from dit_sequence_attention_gb300 import synth
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    per_step = max(0.05, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        cpu_oracle_sample(w, per_step / 4, seed_offset=i)
    flops, secs = 0.0, 0.0
    desc, threads = "", 0
    for i in range(args.steps):
        f, dt, desc, threads = cpu_oracle_sample(w, per_step, seed_offset=100 + i)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.P),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, P):
    return {"workload": f"{w.name}-like packed sequence: {w.n_video} video tokens "
                        f"({w.frames}x{w.grid_h}x{w.grid_w}) + {w.n_audio} audio tokens, padded to {w.S} "
                        f"with masked keys; 56 heads x 128; QK-norm+RoPE -> Ulysses seq2head (P={P}) -> "
                        f"attention per head group -> head2seq",
            "S": w.S, "S_valid": w.S_v, "heads": w.H, "head_dim": w.D, "batch_per_gpu": 1,
            "ulysses_P": P, "l2": f"inputs larger than L2 ({w.S * w.H * w.D * 2 / 1e6:.0f} MB per tensor); no flush"}


class StepRunner:
    """The bench step on one workload's buffers: fused QK-norm+RoPE+seq2head of
    q and k, seq2head of v, one attention launch per head group, head2seq.
    Records CUDA events around each launch on the launching stream."""

    def __init__(self, h3, w, P, q, k, v, wq, wk, pos, stream):
        self.h3, self.w, self.P = h3, w, P
        self.q, self.k, self.v, self.wq, self.wk, self.pos = q, k, v, wq, wk, pos
        self.stream = stream
        self.work = h3.make_workspace(w.S, w.H, w.D, P, q.device)
        self.ev = {"norm": [], "s2h": [], "attn": [], "h2s": []}

    def _mark(self):
        import torch
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def step(self, record=False):
        h3, w, P, work = self.h3, self.w, self.P, self.work
        mark = self._mark if record else (lambda: None)
        e0 = mark()
        h3.h3attn_qk_norm_rope_seq2head(self.q, self.k, work["qh"], work["kh"], self.wq, self.wk, self.pos, P,
                                        *w.rope_split, w.eps, w.theta, stream=self.stream)
        e1 = mark()
        h3.h3attn_seq2head(self.v, work["vh"], P, self.stream)
        e2 = mark()
        marks = []
        for g in range(P):
            h3.h3attn_forward(work["qh"][g], work["kh"][g], work["vh"][g], work["oh"][g], kv_len=w.S_v,
                              stream=self.stream)
            marks.append(mark())
        h3.h3attn_head2seq(work["oh"], work["o"], P, self.stream)
        e4 = mark()
        if record:
            self.ev["norm"].append((e0, e1))
            self.ev["s2h"].append((e1, e2))
            prev = e2
            for m in marks:
                self.ev["attn"].append((prev, m))
                prev = m
            self.ev["h2s"].append((marks[-1], e4))

    def avg_ms(self, name):
        xs = [a.elapsed_time(b) for a, b in self.ev[name]]
        return sum(xs) / len(xs)

    def launches_per_step(self):
        return 1 + 1 + self.P + 1


def timed_region(runner, steps, warmup, world, dev, local, barrier):
    """W untimed steps, then exactly `steps` steps between CUDA events on the
    launching stream, bracketed by a barrier and a device synchronisation on
    both sides, with nvidia-smi clock sampling during the timed steps.
    Returns (max-over-ranks elapsed ms, clock summary)."""
    import torch
    h3 = runner.h3
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize(dev)
    if h3.h3attn_get_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(runner.stream)
    for _ in range(steps):
        runner.step(record=True)
    t_end.record(runner.stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    status = h3.h3attn_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return max_over_ranks(t_start.elapsed_time(t_end), world, dev), clk


def attention_roofline(w, P, attn_ms, peaks, peak_src, clk, n_sm):
    """Roofline of one attention launch (one head group): algorithmic flops
    4 * S_v^2 * D * (H / P) over its CUDA-event duration, against the measured
    dense bf16 burst peak (the sustained figure beside it)."""
    flops_launch = w.attention_flops(heads=w.H // P)
    achieved = flops_launch / (attn_ms * 1e-3) / 1e12
    clock_peak = (n_sm * BF16_FLOP_PER_CLK_SM * clk["sm_mhz"] * 1e6 / 1e12) if clk else None
    return {"kernel": f"attn_fwd_kernel<{w.D}> (one {w.H // P}-head group launch)",
            "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"{peak_src} bf16 dense, burst",
            "sustained_peak": peaks["bf16_tflops_sustained"],
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
            "algorithmic_flops_per_launch": flops_launch, "ms_per_launch": attn_ms,
            "tensor_peak_at_median_clock": clock_peak,
            "frac_of_tensor_peak_at_median_clock": (achieved / clock_peak) if clock_peak else None}


def hbm_kernels(runner, peaks):
    w = runner.w
    tensor_bytes = w.S * w.H * w.D * 2
    ks = {"qk_norm_rope_seq2head": ("norm", 4), "seq2head_v": ("s2h", 2), "head2seq": ("h2s", 2)}
    out = {}
    for name, (ev, mult) in ks.items():
        ms = runner.avg_ms(ev)
        gbs = mult * tensor_bytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "GB_per_s": gbs, "algorithmic_bytes": mult * tensor_bytes,
                     "frac_of_hbm_peak": gbs / peaks["hbm_gbs"], "frac_of_hbm_spec": gbs / HBM_SPEC_GBS}
    return out


def make_inputs(w, dev, rank):
    """Seeded N(0,1) q, k, v of this rank's own sequence (pad rows zero)."""
    from dit_sequence_attention_gb300 import synth
    return tuple(synth.randn_bf16((w.S, w.H, w.D), seed + 1000 * rank, dev, zero_rows_from=w.S_v)
                 for seed in (synth.SEED_Q, synth.SEED_K, synth.SEED_V))


def run_ulysses_across_ranks(args, world, rank, local):
    """--ulysses: one packed sequence split over the N ranks (rows
    [r*S/N, (r+1)*S/N) on rank r), one step = the distributed Ulysses step of
    every rank (all-to-all or all-gather form); `value` = the sequence's
    attention TFLOP/s over the max-over-ranks time (strong scaling).  A single
    process runs it as a one-rank group, which times the collective path."""
    import datetime
    import socket
    import torch
    import torch.distributed as dist
    import dit_sequence_attention_gb300 as h3
    from dit_sequence_attention_gb300 import synth
    from dit_sequence_attention_gb300.ulysses import UlyssesGroup

    h3.load_library()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world == 1:
        os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                timeout=datetime.timedelta(seconds=300))
    g = UlyssesGroup()
    P = g.P
    w = synth.WORKLOADS[args.workload]
    S, H, D = w.S, w.H, w.D
    if S % (P * P) or H % P:
        raise SystemExit(f"--ulysses needs P={P} to divide H and S/P (S={S}, H={H})")
    S_loc = S // P
    rows = slice(g.rank * S_loc, (g.rank + 1) * S_loc)
    wq, wk = (t.to(dev) for t in synth.norm_weights(D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(dev)
    stream = torch.cuda.current_stream(dev)
    if args.ulysses == "a2a":
        q, k, v = (t[rows].contiguous() for t in synth.qkv(w, dev))   # the same sequence on every rank
        pos_loc = pos[rows].contiguous()
        work = g.make_workspace(S_loc, H, D, dev)

        def step():
            g.attention_step(q, k, v, wq, wk, pos_loc, w.S_v, *w.rope_split, w.eps, w.theta, work=work,
                             stream=stream)
        # each rank receives (P-1)/P of its head group's q, k, v rows and of its output rows
        recv_bytes = (3 + 1) * S_loc * H * D * 2 * (P - 1) // P
    else:
        hidden = synth.HIDDEN
        x = synth.fp8_e4m3_codes((S, hidden), 61, 1.0, dev)[rows].contiguous()
        wt = synth.fp8_e4m3_codes((3 * H * D, hidden), 62, 4.0, dev)
        sc = 1.0 / (4.0 * hidden ** 0.5)
        work = g.make_workspace(S_loc, H, D, dev, hidden=hidden)

        def step():
            g.attention_step_allgather(x, wt, sc, wq, wk, pos, w.S_v, *w.rope_split, w.eps, w.theta, work=work,
                                       stream=stream)
        # each rank receives the other ranks' fp8 hidden rows and (P-1)/P of its output rows
        recv_bytes = (P - 1) * S_loc * hidden + S_loc * H * D * 2 * (P - 1) // P
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if h3.h3attn_get_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clk = clocks.stop()
    if h3.h3attn_get_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    t = a.elapsed_time(b)
    tt = torch.tensor([t], dtype=torch.float64, device=dev)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    ms = float(tt.item())
    dist.destroy_process_group()
    if rank != 0:
        return
    value = w.attention_flops() * args.steps / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v or fp8 hidden, random-init "
        "weights)",
        "config": dict(workload_config(w, P), exchange=args.ulysses, parallelism=f"ulysses{P}",
                       received_bytes_per_rank_per_step=recv_bytes),
        "tokens_per_s": w.S_v * args.steps / (ms * 1e-3),
        "clocks": clk,
        "gpu_launches": args.steps * 4,   # this library's kernels per step (the collectives are NCCL's)
        "note": "one sequence over all ranks; every rank's step includes its collectives (NCCL)",
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.ulysses is not None:
        run_ulysses_across_ranks(args, world, rank, local)
        return
    import torch
    import dit_sequence_attention_gb300 as h3
    from dit_sequence_attention_gb300 import synth

    h3.load_library()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    P = args.P
    S, H, D = w.S, w.H, w.D
    # each rank draws its own sequence (independent problems, weak scaling)
    q, k, v = make_inputs(w, dev, rank)
    wq, wk = (t.to(dev) for t in synth.norm_weights(D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(dev)
    stream = torch.cuda.current_stream(dev)
    runner = StepRunner(h3, w, P, q, k, v, wq, wk, pos, stream)
    work = runner.work

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    elapsed_ms, clk = timed_region(runner, args.steps, args.warmup, world, dev, local, barrier)
    flops_seq = w.attention_flops()
    value = job_tflops(flops_seq, args.steps, world, elapsed_ms)
    ms_step = elapsed_ms / args.steps
    attn_ms = runner.avg_ms("attn")                         # per launch (one head group)
    peaks, peak_src = load_peaks()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    roofline = attention_roofline(w, P, attn_ms, peaks, peak_src, clk, n_sm)
    traffic, traffic_src = read_traffic() if (P == 2 and w.name == "480p" and D == 128) else (None, None)
    roofline["traffic"] = traffic
    roofline["traffic_source"] = traffic_src
    roofline["attention_sources_sha256_16"] = attention_fingerprint()
    kernels = hbm_kernels(runner, peaks)
    kernels["attention_per_group"] = {"ms": attn_ms, "TFLOP_per_s": roofline["achieved"]}
    tensor_bytes = S * H * D * 2

    # ---------------------------------------------------------------- e2e
    # Through the public API from pinned host buffers: every step copies its
    # q, k, v and positions host->device and its output device->host.  The two
    # directions run on streams of their own, double-buffered, so the inputs of
    # step i+1 arrive and the output of step i-1 leaves while step i computes
    # (as a streaming caller would).
    e2e_steps = args.e2e_steps or max(2, args.steps)   # the same stream length as the device-timed region
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hpos = pos.cpu().pin_memory()
    hout = [torch.empty((S, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dins = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(pos))
            for _ in range(2)]
    works = [work, h3.make_workspace(S, H, D, P, dev)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def fetch(b):
        for t_dev, t_host in zip(dins[b], (hq, hk, hv, hpos)):
            t_dev.copy_(t_host, non_blocking=True)
        ev_in[b].record(h2d_s)

    def e2e_run(n, ev_first=None):
        for b in range(2):
            ev_out[b].record(d2h_s)             # both output buffers are free
        with torch.cuda.stream(h2d_s):
            if ev_first is not None:
                ev_first.record(h2d_s)
            fetch(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                nb = (i + 1) % 2
                with torch.cuda.stream(h2d_s):
                    if i >= 1:
                        h2d_s.wait_event(ev_done[nb])   # step i-1 finished reading these inputs
                    fetch(nb)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])                 # the output of step i-2 has left this buffer
            dq_, dk_, dv_, dp_ = dins[b]
            o = h3.ulysses_attention_step(dq_, dk_, dv_, wq, wk, dp_, P, w.S_v, *w.rope_split, w.eps, w.theta,
                                          work=works[b], stream=stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[b])
                hout[b].copy_(o, non_blocking=True)
                ev_out[b].record(d2h_s)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    time.sleep(0.3)
    barrier()
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, ev_first=ev_a)       # ev_a: before the first input copy
    ev_b.record(d2h_s)                      # after the last output copy (which follows every step)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_clk = e2e_clocks.stop()
    if h3.h3attn_get_device_status() != 0:
        raise RuntimeError("device status error in the end-to-end loop")
    e2e_ms = max_over_ranks(ev_a.elapsed_time(ev_b), world, dev)
    e2e_value = job_tflops(flops_seq, e2e_steps, world, e2e_ms)
    h2d = 3 * tensor_bytes + hpos.numel() * 4
    d2h = tensor_bytes

    def copy_gbs(dst, src, st):
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            ea.record(st)
            dst.copy_(src, non_blocking=True)
            eb.record(st)
        torch.cuda.synchronize(dev)
        return src.numel() * src.element_size() / (ea.elapsed_time(eb) * 1e-3) / 1e9
    link = {"h2d_GB_per_s": copy_gbs(dins[0][0], hq, h2d_s), "d2h_GB_per_s": copy_gbs(hout[0], works[0]["o"], d2h_s)}
    del hq, hk, hv, hout, dins, works

    # --------------------------------------- the 262k end of the metric: 1080p
    # A short leg on the 1080p-like sequence (262,144 tokens) with the same
    # step and launch configuration, timed the same way; the headline above
    # stays on the bench workload.
    long_leg = None
    if args.long_steps > 0 and w.name != "1080p" and D == 128:
        wl = synth.WORKLOADS["1080p"]
        ql, kl, vl = make_inputs(wl, dev, rank)
        posl = torch.from_numpy(synth.packed_positions(wl)).to(dev)
        rl = StepRunner(h3, wl, P, ql, kl, vl, wq, wk, posl, stream)
        el_ms, clk_l = timed_region(rl, args.long_steps, args.long_warmup, world, dev, local, barrier)
        ms_l = el_ms / args.long_steps
        long_leg = {
            "1080p": {"config": workload_config(wl, P), "steps": args.long_steps, "warmup": args.long_warmup,
                      "ms_per_step": ms_l, "value": job_tflops(wl.attention_flops(), args.long_steps, world, el_ms),
                      "unit": "TFLOP/s",
                      "tokens_per_s": wl.S_v * args.long_steps * world / (el_ms * 1e-3),
                      "roofline": attention_roofline(wl, P, rl.avg_ms("attn"), peaks, peak_src, clk_l, n_sm),
                      "kernels": hbm_kernels(rl, peaks), "clocks": clk_l,
                      "gpu_launches": args.long_steps * rl.launches_per_step()}}
        del ql, kl, vl, rl

    # ------------------------------- head-chunked attention, overlapped exchange
    # The same step with each group's heads split into chunks; the output
    # exchange of chunk c runs on a second stream while attention computes
    # chunk c+1 (bit-identical output for any chunk count).
    chunk_runs = None
    if not args.no_chunks:
        xs = torch.cuda.Stream(dev)
        chunk_runs = {"chunks": [1], "ms_per_step": [ms_step], "attention_launches_per_step": [P]}
        ref_out = h3.ulysses_attention_step(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps, w.theta,
                                            work=work, stream=stream).clone()
        for c in (2, 4):
            def chunked_step():
                return h3.ulysses_attention_step(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps, w.theta,
                                                  work=work, stream=stream, attn_chunks=c, exchange_stream=xs)
            for _ in range(2):
                chunked_step()
            torch.cuda.synchronize(dev)
            ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_c = max(3, min(args.steps, 6))
            ca.record(stream)
            for _ in range(n_c):
                out_c = chunked_step()
            cb.record(stream)  # the step joins the exchange stream back into `stream` before returning
            torch.cuda.synchronize(dev)
            if h3.h3attn_get_device_status() != 0:
                raise RuntimeError("device status error in the chunked step")
            if not torch.equal(out_c.view(torch.int16), ref_out.view(torch.int16)):
                raise RuntimeError(f"chunked step ({c} chunks) is not bit-identical to the unchunked one")
            chunk_runs["chunks"].append(c)
            chunk_runs["ms_per_step"].append(ca.elapsed_time(cb) / n_c)
            chunk_runs["attention_launches_per_step"].append(P * c)
        chunk_runs["note"] = ("whole step; output exchange of each head chunk on a second stream, overlapping the "
                              "next chunk's attention; outputs checked bit-identical to the unchunked step")
        del ref_out

    # ------------------------------------------------ whole step as a CUDA graph
    graph_runs = None
    if args.graph and D == 128:
        sg = h3.StepGraph(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps, w.theta)
        gwork = h3.make_workspace(S, H, D, P, dev)
        n_g = max(3, min(args.steps, 20))

        def timed(fn, n):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(stream)
            for _ in range(n):
                fn()
            gb.record(stream)
            torch.cuda.synchronize(dev)
            return ga.elapsed_time(gb) / n

        eager_ms = timed(lambda: h3.ulysses_attention_step(q, k, v, wq, wk, pos, P, w.S_v, *w.rope_split, w.eps,
                                                           w.theta, work=gwork, stream=stream), n_g)
        graph_ms = timed(sg.replay, n_g)
        if h3.h3attn_get_device_status() != 0:
            raise RuntimeError("device status error in the graph timing")
        if not torch.equal(sg.out.view(torch.int16), gwork["o"].view(torch.int16)):
            raise RuntimeError("graph replay differs from the eager step")
        graph_runs = {"eager_ms_per_step": eager_ms, "graph_ms_per_step": graph_ms, "steps": n_g}
        del sg, gwork

    # ---------------------------------------------- all-gather variant projection
    proj = None
    if not args.no_proj and D == 128:
        hidden, inner = synth.HIDDEN, synth.INNER
        xg = synth.fp8_e4m3_codes((S, hidden), 41 + rank, 1.0, dev)
        wg = synth.fp8_e4m3_codes((3 * inner, hidden), 42, 4.0, dev)
        outs = [torch.empty((S, inner // P), dtype=torch.bfloat16, device=dev) for _ in range(3)]
        sc = 1.0 / (4.0 * hidden ** 0.5)
        for _ in range(3):
            h3.h3attn_qkv_proj_fp8(xg, wg, sc, *outs, P, 0)
        torch.cuda.synchronize(dev)
        pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        pa.record(stream)
        for _ in range(reps):
            h3.h3attn_qkv_proj_fp8(xg, wg, sc, *outs, P, 0)
        pb.record(stream)
        torch.cuda.synchronize(dev)
        if h3.h3attn_get_device_status() != 0:
            raise RuntimeError("device status error in the projection timing")
        pms = pa.elapsed_time(pb) / reps
        pfl = 2.0 * S * (3 * inner // P) * hidden
        fp8_peak = 2.0 * peaks["bf16_tflops"]
        proj = {"kernel": "qkv_proj_fp8_kernel (one rank of P)", "shape": f"[{S} x {hidden}] x [{hidden} x 3*{inner}/{P}]",
                "ms": pms, "TFLOP_per_s": pfl / (pms * 1e-3) / 1e12,
                "peak": fp8_peak, "peak_source": f"{peak_src} bf16 burst x 2 (dense fp8 / bf16 nominal ratio)",
                "frac": pfl / (pms * 1e-3) / 1e12 / fp8_peak}
        del xg, wg, outs
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        f, dt, desc, threads = cpu_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
               "sample_seconds": dt,
               "extrapolated_full_step_s": w.attention_flops() / (f / dt),
               "note": "extrapolated: the whole 56-head step at the sample's measured rate"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v, random-init norm weights)",
        "config": workload_config(w, P),
        "tokens_per_s": w.S_v * args.steps * world / (elapsed_ms * 1e-3),
        "frac_of_bf16_peak": value / peaks["bf16_tflops"],
        "padded_work_tflops": value * S / w.S_v,
        "padded_work_note": "the same step counted as 4*S*S_v*D*H (every padded query row against the valid keys)",
        "roofline": roofline,
        "kernels": kernels,
        "hbm_peak_GB_per_s": peaks["hbm_gbs"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps, "copy_link": link, "clocks": e2e_clk,
                "note": "pinned host q/k/v/pos -> device, whole path, device -> pinned host output each step; "
                        "each direction double-buffered on its own stream, overlapping compute; copy_link = one "
                        "734 MB copy each way measured alone"},
        "gpu_launches": args.steps * runner.launches_per_step(),
        "clocks": clk,
        "workloads": long_leg,
        "cpu_baseline": cpu,
        "ag_qkv_proj_fp8": proj,
        "head_chunk_overlap": chunk_runs,
        "cuda_graph": graph_runs,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
