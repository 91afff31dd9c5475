#!/usr/bin/env python
"""Benchmark of the KDA recurrence library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the hot path on one batch of seeded synthetic input
already resident in HBM:
  varlen_64k         kda_prefill_chunked over 8 packed sequences (65536 tokens)
                     with S0, then kda_decode_step for all 8 (default: the
                     largest workload)
  prefill_32k_carry  kda_prefill_chunked, H=96, T=32768 with S0
  prefill_4k         kda_prefill_chunked, H=96, T=4096, bf16 q/k/v, chunk 64
  tiny_fp32          kda_prefill_chunked, H=2, T=64, fp32 q/k/v, chunk 16
                     (the CUDA-core path)
The JSON line's value is prefill tokens/s of the headline workload; the
other prefill workloads are reported under "legs", each with its roofline.
The metric's second half, decode state GB/s, is measured on the batched
decode workload (B=64, H=96, 100 consecutive in-place steps) and reported
under "decode".

Inputs (and outputs) exceed the 129 MB L2, so no L2 flush is done between
steps.  Timing: CUDA events on the launching stream, W untimed warm-up steps,
then exactly K timed steps between a barrier and a device synchronise on both
sides; max over ranks.  Under torchrun each rank runs an independent replica
on its own GPU (the path has no cross-GPU exchange): weak scaling.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kda_inputs as ki  # noqa: E402

METRIC = "KDA prefill tokens/s (% BF16 TC peak); decode state GB/s (% of 8 TB/s HBM)"
UNIT = "tokens/s"
DK = DV = 128
# algorithmic bytes per token-head of a prefill: q, k, v bf16 (3 x 256) + g fp32
# (512) + beta (4) + o fp32 (512)
PREFILL_BYTES_PER_TOKEN_HEAD_BF16 = 3 * 256 + 512 + 4 + 512
STATE_BYTES = DK * DV * 4
# flops per token-head of the chunked form with chunk C: 2C(3dk + 2dv) + 6 dk dv
def prefill_flops_per_token_head(C):
    return 2 * C * (3 * DK + 2 * DV) + 6 * DK * DV
# algorithmic bytes per (b, h) of a decode step: state read + write, q, k, v bf16,
# g fp32, beta, o fp32
DECODE_BYTES_PER_STATE = 2 * STATE_BYTES + 3 * 256 + 512 + 4 + 512
FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12   # fp32 FMA lanes x 2 flop x max SM clock


def code_sha(source_file):
    """sha256 prefix of a kernel source's code: comments removed and
    whitespace collapsed, so that edits to comments keep a capture valid."""
    import hashlib
    import re
    src = open(os.path.join(ROOT, "kda_linear_attention_gb300", "csrc", source_file)).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()[:16]


TRAFFIC_FILE = os.path.join("profiles", "dram_traffic.json")


def _traffic(kernel, source_file):
    """DRAM bytes per launch of `kernel` as stored from an ncu capture in
    profiles/dram_traffic.json, if that capture was taken on the current
    kernel code (code_sha), else None.  A stored capture, not a number
    measured by this run."""
    rec = _traffic_record(kernel, source_file)
    return None if rec is None else int(rec["bytes"])


def _traffic_record(kernel, source_file):
    try:
        sha = code_sha(source_file)
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as f:
            data = json.load(f)
        for rec in data.get("captures", []):
            if rec.get("kernel") == kernel and rec.get("code_sha256") == sha:
                return rec
    except Exception:
        pass
    return None


def _prefill_traffic(units):
    """DRAM bytes of one tensor-core prefill call over `units` (chunk, head)
    pairs, from the stored captures of its two kernels scaled by units (both
    kernels' traffic is per (chunk, head): records, q/k/g/beta/v in, o out),
    with a note of where the number comes from; (None, reason) if there is
    no capture on the current code."""
    recs = [_traffic_record(k, "kda_prefill_split.cu") for k in ("intra_chunk_kernel", "state_pass_kernel")]
    if None in recs:
        return None, "no stored capture on the current kernel code"
    tot = 0.0
    for r in recs:
        tot += r["bytes"] * units / r["units"]
    src = "stored ncu capture (%s, %s), dram__bytes_read.sum + dram__bytes_write.sum" % (
        TRAFFIC_FILE, recs[0].get("workload"))
    if units != recs[0]["units"]:
        src += ", scaled by (chunk, head) units %d -> %d" % (recs[0]["units"], units)
    return int(round(tot)), src


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling (every 200 ms) around the timed
    region.  The timed steps of a workload last only milliseconds, so the
    sampler is started first and the GPU is kept busy with untimed steps of
    the same workload until samples arrive (``keep_busy``) before and after
    the timed steps: the load window the samples cover contains the timed
    region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self._lock = threading.Lock()
        self._reader = None

    def _read(self):
        for line in self.proc.stdout:
            with self._lock:
                self.lines.append(line)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception:
            self.proc = None
        return self

    def count(self) -> int:
        with self._lock:
            return len(self.lines)

    def keep_busy(self, step, n_new: int, timeout_s: float = 5.0, batch: int = 16):
        """Run untimed steps (batches of `batch`, then a device synchronise)
        until `n_new` more samples have arrived, for at most `timeout_s`."""
        import torch
        if self.proc is None:
            return
        target = self.count() + n_new
        t_end = time.monotonic() + timeout_s
        while self.count() < target and time.monotonic() < t_end:
            for _ in range(batch):
                step()
            torch.cuda.synchronize()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._reader is not None:
                self._reader.join(timeout=5)

    def summary(self):
        rows = []
        with self._lock:
            lines = list(self.lines)
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]),
                                 hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows),
                "window": "every 200 ms over a load window of untimed steps of the same "
                          "workload that contains the timed steps"}


# ---------------------------------------------------------------------------
def _gpu_hold(torch, ms: float):
    """Keep the GPU busy for about `ms` milliseconds (a bounded spin kernel)
    while the host enqueues the timed launches behind it: a timed region
    then measures device time only, never the host's call overhead."""
    torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time: every rank's timed region covers the same
    per-rank work (a replica), so the job takes as long as its slowest rank."""
    if ws <= 1:
        return ms
    import torch
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(units_per_rank: float, ws: int, ms: float) -> float:
    """Whole-job units per second: every rank processed units_per_rank in
    the (max-over-ranks) time ms."""
    return ws * units_per_rank / (ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _pinned(a):
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


PREFILL_WORKLOADS = ["varlen_64k", "prefill_32k_carry", "prefill_4k", "tiny_fp32"]
REC_BYTES = 60416          # per-(chunk, head) record of the two-kernel tensor-core prefill


class PrefillCase:
    """One prefill workload resident on the device, ready to be stepped."""

    def __init__(self, kda, torch, dev, wl):
        self.kda, self.torch, self.wl = kda, torch, wl
        if wl == "varlen_64k":
            pre, dstep = ki.workload_varlen_with_decode(wl)
        else:
            pre, dstep = ki.workload_prefill(wl), None
        self.pre, self.dstep = pre, dstep
        self.T, self.H, self.N, self.C = pre.T, pre.H, pre.N, pre.chunk
        self.d = {n: _to_dev(getattr(pre, n), dev) for n in ("q", "k", "v", "g", "beta")}
        self.cu = _to_dev(pre.cu_seqlens, dev)
        self.S0 = None if pre.S0 is None else _to_dev(pre.S0, dev)
        self.o = torch.empty((self.T, self.H, DV), dtype=torch.float32, device=dev)
        self.S_out = torch.empty((self.N, self.H, DK, DV), dtype=torch.float32, device=dev)
        if dstep is not None:
            self.dd = {n: _to_dev(getattr(dstep, n), dev) for n in ("q", "k", "v", "g", "beta")}
            self.od = torch.empty((self.N, self.H, DV), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # tensor-core path: chunk plan + intra-chunk kernel + state pass per call
        self.tc = pre.dtype == "bf16" and self.C == 64 and self.T > 0
        self.launches = (3 if self.tc else 1) + (1 if dstep is not None else 0)
        self.ev = []

    def step(self, record=False):
        kda, torch, d = self.kda, self.torch, self.d
        if record and self.tc:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            kda.prefill_chunked_events(d["q"], d["k"], d["v"], d["g"], d["beta"], self.cu, evs,
                                       S0=self.S0, o=self.o, S_out=self.S_out)
            self.ev.append(evs)
        else:
            if record:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
            kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], self.cu, S0=self.S0,
                                chunk=self.C, o=self.o, S_out=self.S_out)
            if record:
                b.record(self.stream)
                self.ev.append([a, b])
        if self.dstep is not None:
            x = self.dd
            kda.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], self.S_out, o=self.od)

    def kernel_ms(self):
        """Mean prefill time per call (first to last event) and, on the
        tensor-core path, per kernel (plan, intra-chunk, state pass)."""
        kern = statistics.mean(e[0].elapsed_time(e[-1]) for e in self.ev)
        parts = None
        if self.tc:
            parts = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in self.ev) for i in range(3)]
        return kern, parts

    def roofline(self, peaks):
        pre, T, H, N, C = self.pre, self.T, self.H, self.N, self.C
        kern_ms, part_ms = self.kernel_ms()
        tok_heads = T * H
        n_state = N * H
        per_th = PREFILL_BYTES_PER_TOKEN_HEAD_BF16 if pre.dtype == "bf16" else (3 * 512 + 512 + 4 + 512)
        alg_bytes = tok_heads * per_th + n_state * STATE_BYTES * (2 if self.S0 is not None else 1)
        alg_flops = tok_heads * prefill_flops_per_token_head(C)
        achieved_gbs = alg_bytes / (kern_ms / 1e3) / 1e9
        achieved_tflops = alg_flops / (kern_ms / 1e3) / 1e12
        hbm_frac = achieved_gbs / peaks["hbm"]
        tc_frac = achieved_tflops / peaks["bf16"]
        if self.tc:
            # Designed against the HBM roofline (arithmetic intensity ~100
            # flop/B, below the bf16 ridge point).  One call = chunk plan +
            # intra-chunk kernel + state pass; its roofline is the call's
            # (algorithmic bytes / call time: the per-chunk records the two
            # kernels exchange count against it), and each kernel is reported
            # with the bytes it moves in this design.
            lens = np.diff(pre.cu_seqlens)
            nchunk = int(sum((int(x) + 63) // 64 for x in lens))
            intra_bytes = nchunk * H * (2 * 64 * 256 + 64 * 512 + 64 * 4 + REC_BYTES)
            state_bytes = nchunk * H * (REC_BYTES + 64 * 256) + T * H * 512 + n_state * STATE_BYTES * (
                2 if self.S0 is not None else 1)
            kernels = {}
            for kname, ms_k, mb in (("chunk_plan_kernel", part_ms[0], None),
                                    ("intra_chunk_kernel", part_ms[1], intra_bytes),
                                    ("state_pass_kernel", part_ms[2], state_bytes)):
                kd = {"ms": round(ms_k, 4), "share": round(ms_k / kern_ms, 4)}
                if mb is not None:
                    kd.update({"moved_bytes": int(mb), "gbs": round(mb / (ms_k / 1e3) / 1e9, 1),
                               "frac_hbm": round(mb / (ms_k / 1e3) / 1e9 / peaks["hbm"], 4)})
                kernels[kname] = kd
            traffic, tsrc = _prefill_traffic(nchunk * H)
            roof = {
                "kernel": "prefill call: chunk_plan_kernel + intra_chunk_kernel + state_pass_kernel "
                          "(tcgen05/TMEM/TMA); dominant: intra_chunk_kernel",
                "bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm"],
                "unit": "GB/s", "frac": round(hbm_frac, 4), "of": peaks["source"],
                "traffic": traffic, "traffic_source": tsrc,
                "kernels": kernels,
            }
        else:
            roof = {
                "kernel": "prefill_simt_kernel (fp32 CUDA-core chunked prefill)",
                "bound": "alu", "achieved": round(achieved_tflops, 4),
                "peak": round(FFMA_PEAK_TFLOPS, 1), "unit": "TFLOP/s",
                "frac": round(achieved_tflops / FFMA_PEAK_TFLOPS, 5),
                "of": "derived: 152 SMs x 128 FMA lanes x 2 flop x 2.07 GHz", "traffic": None,
            }
        roof.update({
            "tensor": {"achieved_tflops": round(achieved_tflops, 2), "peak_tflops": peaks["bf16"],
                       "frac": round(tc_frac, 5), "of": peaks["source"]},
            "hbm": {"achieved_gbs": round(achieved_gbs, 1), "peak_gbs": peaks["hbm"],
                    "frac": round(hbm_frac, 5), "of": peaks["source"]},
            "kernel_ms": round(kern_ms, 4),
            "algorithmic_bytes": int(alg_bytes), "algorithmic_flops": int(alg_flops),
            "bytes_per_token_head": per_th, "flops_per_token_head": prefill_flops_per_token_head(C),
        })
        return roof

    def config(self):
        pre = self.pre
        return {"workload": self.wl, "H": self.H, "T": self.T, "N": self.N, "chunk": self.C,
                "dk": DK, "dv": DV, "qkv": pre.dtype, "S0": self.S0 is not None,
                "lens": [int(x) for x in np.diff(pre.cu_seqlens)] if self.N > 1 else None,
                "then_decode": self.dstep is not None}


def _leg(case, peaks, reps):
    """A secondary prefill workload: `reps` calls back to back behind a GPU
    hold (median call time and per-kernel times from CUDA events), with its
    roofline."""
    torch = case.torch
    for _ in range(3):
        case.step()
    torch.cuda.synchronize()
    case.ev = []
    _gpu_hold(torch, 3.0 * reps)
    for _ in range(reps):
        case.step(record=True)
    torch.cuda.synchronize()
    med = statistics.median(e[0].elapsed_time(e[-1]) for e in case.ev)
    roof = case.roofline(peaks)
    return {"config": case.config(), "ms_per_call": round(med, 4),
            "tokens_per_s": round(case.T / (med / 1e3), 1), "calls": reps,
            "gpu_launches_per_call": case.launches, "roofline": roof}


def run_ours(args):
    import torch
    import kda_linear_attention_gb300 as kda
    from kda_linear_attention_gb300 import build as kbuild

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws > 1:
        kbuild.build()
    if ws > 1:
        torch.distributed.barrier()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    wl = args.workload
    case = PrefillCase(kda, torch, dev, wl)
    stream = case.stream
    for _ in range(args.warmup):
        case.step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.keep_busy(case.step, 2)        # untimed load until the sampler reports
        barrier()
        torch.cuda.synchronize()
        _gpu_hold(torch, 3.0 * args.steps * max(1.0, case.T / 4096))
        t0.record(stream)
        for _ in range(args.steps):
            case.step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
        clk.keep_busy(case.step, 1)
    barrier()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    ms_per_step = ms / args.steps
    value = job_throughput(case.T, ws, ms_per_step)
    peaks = _peaks()
    roofline = case.roofline(peaks)
    config = case.config()
    config.update({"l2": "inputs larger than L2 (no flush)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"})
    dstep = case.dstep

    # ---- the other prefill workloads, each with its roofline --------------
    legs = {}
    if not args.no_legs:
        for other in PREFILL_WORKLOADS:
            if other == wl:
                continue
            c2 = PrefillCase(kda, torch, dev, other)
            legs[other] = _leg(c2, peaks, reps=max(5, args.steps))
            del c2
            torch.cuda.empty_cache()

    # ---- decode leg: B=64, H=96, 100 consecutive in-place steps ----------
    decode = None
    if not args.no_decode:
        decode = _decode_leg(kda, torch, dev, stream, peaks, args)

    # ---- the layer around the recurrence (prologue, gated epilogue, fused decode)
    layer = None
    if not args.no_layer:
        layer = _layer_leg(kda, torch, dev, stream, peaks)

    # ---- end to end through the public API with host buffers -------------
    e2e = None if args.no_e2e else _e2e_leg(kda, torch, dev, stream, case.pre, dstep, args, barrier, ws)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 state/accumulate" if case.pre.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and distributions of the model's KDA layer)",
        "config": config,
        "gpu_launches": case.launches * args.steps,
        "roofline": roofline,
        "legs": legs or None,
        "decode": decode,
        "layer": layer,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(case.pre, args)
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _decode_leg(kda, torch, dev, stream, peaks, args):
    w = ki.WORKLOADS["decode_b64"]
    B, H, n_steps = w["B"], w["H"], w["steps"]
    S_np, steps = ki.workload_decode("decode_b64")
    S = _to_dev(S_np, dev)
    steps = iter(steps)
    first = next(steps)
    cpu = None if args.no_cpu_baseline else _decode_cpu_baseline(S_np, first, B, H)
    del S_np
    ins = [{n: _to_dev(getattr(st, n), dev) for n in ("q", "k", "v", "g", "beta")}
           for st in itertools.chain([first], steps)]
    o = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    for i in range(3):
        x = ins[i]
        kda.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], S, o=o)
    torch.cuda.synchronize()
    evs = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)

    def untimed():
        x = ins[0]
        kda.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], S, o=o)

    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.keep_busy(untimed, 2, batch=64)
        _gpu_hold(torch, 2.0 * len(ins))
        t0.record(stream)
        for x in ins:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            kda.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], S, o=o)
            b.record(stream)
            evs.append((a, b))
        t1.record(stream)
        torch.cuda.synchronize()
        clk.keep_busy(untimed, 1, batch=64)
    per = [a.elapsed_time(b) for a, b in evs]
    total = t0.elapsed_time(t1)
    med = statistics.median(per)
    state_bytes = 2 * STATE_BYTES * B * H
    all_bytes = DECODE_BYTES_PER_STATE * B * H
    gbs_state = state_bytes / (med / 1e3) / 1e9
    gbs_all = all_bytes / (med / 1e3) / 1e9
    return {
        "workload": "decode_b64 (B=64, H=96, 100 consecutive in-place steps)",
        "metric": "decode state GB/s", "value": round(gbs_state, 1), "unit": "GB/s",
        "median_step_us": round(med * 1e3, 2), "total_ms_100_steps": round(total, 3),
        "roofline": {"kernel": "kda_decode", "bound": "hbm", "achieved": round(gbs_all, 1),
                     "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": round(gbs_all / peaks["hbm"], 4), "of": peaks["source"],
                     "frac_of_nominal_8tbs": round(gbs_all / 8000.0, 4),
                     "traffic": _traffic("decode_kernel", "kda_decode.cu"),
                     "algorithmic_bytes": int(all_bytes)},
        "gpu_launches": n_steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "pool_bf16": _decode_pool_leg(kda, torch, dev, stream, peaks, S, ins, B, H),
    }


def _decode_cpu_baseline(S_np, step, B, H):
    """The fp64 oracle on one whole decode step (every state), timed on the
    host cores, in the decode metric (state bytes read and written / s)."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    oracle.decode(S_np[:1], _first_rows(step, 1), threads=threads)     # warm
    t = time.perf_counter()
    oracle.decode(S_np, step, threads=threads)
    dt = time.perf_counter() - t
    state_bytes = 2 * STATE_BYTES * B * H
    return {"value": round(state_bytes / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "one whole decode step (%d states) of the fp64 oracle, %.2f s" % (B * H, dt)}


def _first_rows(step, b):
    """The first b sequences of a decode step (same type, sliced fields)."""
    import copy
    st = copy.copy(step)
    for n in ("q", "k", "v", "g", "beta"):
        setattr(st, n, getattr(step, n)[:b])
    return st


def _timed(torch, stream, fn, reps=10, warm=3):
    """Median CUDA-event time (ms) of fn() on `stream` over `reps` calls,
    enqueued back to back behind a GPU hold (so host-side call overhead
    never leaves the GPU idle between the events)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    _gpu_hold(torch, 2.0 * reps)
    ts = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


# algorithmic bytes of the layer's kernels
PROLOGUE_BYTES_PER_TOKEN_HEAD = 3 * 256 + 3 * 256        # raw q/k/v in, q/k/v out (bf16)
# layer prefill per token-head: raw q/k/v and gate in (bf16), g, beta in,
# the gated output out (fp32); per (sequence, head) the state in and out and
# the conv window in and out
LAYER_PREFILL_BYTES_PER_TOKEN_HEAD = 3 * 256 + 256 + 512 + 4 + 512
# decode layer step per (b, h): state read + write, raw q/k/v, gate (bf16),
# conv window read + write (3 x 3 x 128 bf16 each), g, beta, out (fp32)
DECODE_LAYER_BYTES_PER_STATE = 2 * STATE_BYTES + 3 * 256 + 256 + 2 * 2304 + 512 + 4 + 512


def _layer_leg(kda, torch, dev, stream, peaks):
    """The layer around the recurrence at the model's sizes: the conv1d +
    SiLU + L2-norm prologue and the gated prefill on the 4K prefill (H = 96,
    T = 4096), the fused whole-layer decode step on the batched decode
    (B = 64, H = 96, fp32 state pool, permuted slots)."""
    L = ki.gen_layer(21, [4096], H=96, with_conv0=True)
    T, H = L.T, L.H
    d = {n: _to_dev(getattr(L, n), dev) for n in ("xq", "xk", "xv", "conv_w", "conv0", "gate",
                                                   "norm_w", "g", "beta", "cu_seqlens")}
    q = torch.empty((T, H, DK), dtype=torch.bfloat16, device=dev)
    k, v = torch.empty_like(q), torch.empty_like(q)
    conv_out = torch.empty_like(d["conv0"])
    out = torch.empty((T, H, DV), dtype=torch.float32, device=dev)
    S_out = torch.empty((1, H, DK, DV), dtype=torch.float32, device=dev)

    def prologue():
        kda.conv_prologue(d["xq"], d["xk"], d["xv"], d["conv_w"], d["cu_seqlens"],
                          conv_in=d["conv0"], conv_out=conv_out, q=q, k=k, v=v)

    def gated():
        kda.prefill_chunked_gated(q, k, v, d["g"], d["beta"], d["cu_seqlens"], d["gate"],
                                  d["norm_w"], out=out, S_out=S_out)

    def plain():
        kda.prefill_chunked(q, k, v, d["g"], d["beta"], d["cu_seqlens"], o=out, S_out=S_out)

    def two_calls():
        prologue()
        gated()

    def one_call():
        kda.prefill_layer(d["xq"], d["xk"], d["xv"], d["conv_w"], d["g"], d["beta"], d["gate"],
                          d["norm_w"], d["cu_seqlens"], conv_in=d["conv0"], out=out, S_out=S_out,
                          conv_out=conv_out)

    t_pro = _timed(torch, stream, prologue)
    t_gated = _timed(torch, stream, gated)
    t_plain = _timed(torch, stream, plain)
    t_two = _timed(torch, stream, two_calls)
    t_all = _timed(torch, stream, one_call)
    pro_bytes = T * H * PROLOGUE_BYTES_PER_TOKEN_HEAD
    pro_gbs = pro_bytes / (t_pro / 1e3) / 1e9
    lay_bytes = T * H * LAYER_PREFILL_BYTES_PER_TOKEN_HEAD + H * (STATE_BYTES + 2 * 2304)
    lay_gbs = lay_bytes / (t_all / 1e3) / 1e9
    prefill = {
        "workload": "layer prefill, H=96, T=4096, chunk 64, bf16 raw projections, carried windows",
        "call": "kda_layer_prefill (conv_prologue_kernel, then the gated prefill's three launches)",
        "ms": round(t_all, 4), "tokens_per_s": round(T / (t_all / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(lay_gbs, 1), "peak": peaks["hbm"],
                     "unit": "GB/s", "frac": round(lay_gbs / peaks["hbm"], 4),
                     "algorithmic_bytes": int(lay_bytes),
                     "bytes_per_token_head": LAYER_PREFILL_BYTES_PER_TOKEN_HEAD, "traffic": None},
        "vs_gated_prefill_alone": round(t_all / t_gated, 4),
        "two_calls_ms": round(t_two, 4),
        "prologue": {"kernel": "conv_prologue_kernel", "ms": round(t_pro, 4),
                     "roofline": {"bound": "hbm", "achieved": round(pro_gbs, 1),
                                  "peak": peaks["hbm"], "unit": "GB/s",
                                  "frac": round(pro_gbs / peaks["hbm"], 4),
                                  "algorithmic_bytes": int(pro_bytes),
                                  "bytes_per_token_head": PROLOGUE_BYTES_PER_TOKEN_HEAD,
                                  "traffic": _traffic("conv_prologue_kernel", "kda_layer.cu")}},
        "gated_prefill": {"ms": round(t_gated, 4), "ungated_ms": round(t_plain, 4),
                          "epilogue_overhead_frac": round(t_gated / t_plain - 1.0, 4)},
        "gpu_launches_per_call": 4,
    }
    del L, d, q, k, v, out

    B, Hd = 64, 96
    rng = np.random.Generator(np.random.PCG64(22))
    Ld = ki.gen_layer(23, [1], H=Hd)
    step = ki.gen_layer_decode_step(rng, B, Hd)
    S = torch.from_numpy(ki.gen_decode_state(rng, B, Hd)).to(dev)
    conv = torch.randn((B, 3, 3, Hd, DK), generator=torch.Generator().manual_seed(24)).to(
        torch.bfloat16).to(dev)
    slots = torch.randperm(B, generator=torch.Generator().manual_seed(25)).to(torch.int32).to(dev)
    x = {n: _to_dev(getattr(step, n), dev) for n in ("xq", "xk", "xv", "gate", "g", "beta")}
    w = _to_dev(Ld.conv_w, dev)
    nw = _to_dev(Ld.norm_w, dev)
    o = torch.empty((B, Hd, DV), dtype=torch.float32, device=dev)

    def layer_step():
        kda.decode_layer_step(x["xq"], x["xk"], x["xv"], w, conv, x["g"], x["beta"], x["gate"], nw,
                              S, state_indices=slots, out=o)

    t_step = _timed(torch, stream, layer_step, reps=100)
    plain = ki.gen_decode_step(rng, B, Hd, "bf16")
    y = {n: _to_dev(getattr(plain, n), dev) for n in ("q", "k", "v", "g", "beta")}
    t_dec = _timed(torch, stream, lambda: kda.decode_step_pool(
        y["q"], y["k"], y["v"], y["g"], y["beta"], S, state_indices=slots, o=o), reps=100)
    step_bytes = B * Hd * DECODE_LAYER_BYTES_PER_STATE + 3 * Hd * DK * 4 * 4 + DV * 4
    gbs = step_bytes / (t_step / 1e3) / 1e9
    decode = {
        "workload": "layer decode step, B=64, H=96, fp32 state pool, permuted slots",
        "median_step_us": round(t_step * 1e3, 2),
        "recurrence_only_step_us": round(t_dec * 1e3, 2),
        "roofline": {"kernel": "decode_layer_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": round(gbs / peaks["hbm"], 4),
                     "algorithmic_bytes": int(step_bytes),
                     "bytes_per_state": DECODE_LAYER_BYTES_PER_STATE,
                     "traffic": _traffic("decode_layer_kernel", "kda_layer.cu")},
        "gpu_launches_per_step": 1,
    }
    return {"prefill": prefill, "decode": decode}


def _decode_pool_leg(kda, torch, dev, stream, peaks, S32, ins, B, H):
    """The same 100 steps on a bf16 state pool addressed by a permuted slot
    table (kda_decode_step_pool): half the state bytes per step."""
    P = B
    S = S32.to(torch.bfloat16)
    g = torch.Generator().manual_seed(7)
    slots = torch.randperm(P, generator=g).to(torch.int32).to(dev)
    o = torch.empty((B, H, DV), dtype=torch.float32, device=dev)
    for i in range(3):
        x = ins[i]
        kda.decode_step_pool(x["q"], x["k"], x["v"], x["g"], x["beta"], S, state_indices=slots, o=o)
    torch.cuda.synchronize()
    evs = []
    _gpu_hold(torch, 2.0 * len(ins))
    for x in ins:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kda.decode_step_pool(x["q"], x["k"], x["v"], x["g"], x["beta"], S, state_indices=slots, o=o)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    med = statistics.median(a.elapsed_time(b) for a, b in evs)
    state_bytes = 2 * (STATE_BYTES // 2) * B * H
    all_bytes = (DECODE_BYTES_PER_STATE - STATE_BYTES) * B * H
    gbs_all = all_bytes / (med / 1e3) / 1e9
    return {"workload": "decode_b64 on a bf16 pool, permuted slots", "median_step_us": round(med * 1e3, 2),
            "state_gbs": round(state_bytes / (med / 1e3) / 1e9, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs_all, 1), "peak": peaks["hbm"],
                         "unit": "GB/s", "frac": round(gbs_all / peaks["hbm"], 4),
                         "algorithmic_bytes": int(all_bytes),
                         "traffic": _traffic("decode_bf16_state_kernel", "kda_decode.cu")},
            "gpu_launches": len(ins)}


def _e2e_leg(kda, torch, dev, stream, pre, dstep, args, barrier, ws):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory to the device and reads its outputs
    (o, S_out, and the decode's o) back to pinned host memory.  Steps are
    pipelined the way a serving loop runs them: step i+1's inputs are copied
    in (copy-in stream) while step i computes (compute stream) and step i-1's
    outputs are copied out (copy-out stream), with two sets of device
    buffers; the timed region runs from the first copy-in to the last
    copy-out."""
    names = ("q", "k", "v", "g", "beta")
    host = {n: _pinned(getattr(pre, n)) for n in names}
    cu_h = _pinned(pre.cu_seqlens)
    S0_h = None if pre.S0 is None else _pinned(pre.S0)
    T, H, N = pre.T, pre.H, pre.N
    NB = 2
    o_h = [torch.empty((T, H, DV), dtype=torch.float32).pin_memory() for _ in range(NB)]
    S_h = [torch.empty((N, H, DK, DV), dtype=torch.float32).pin_memory() for _ in range(NB)]
    if dstep is not None:
        dh = {n: _pinned(getattr(dstep, n)) for n in names}
        od_h = [torch.empty((N, H, DV), dtype=torch.float32).pin_memory() for _ in range(NB)]
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + cu_h.numel() * 4
    h2d += 0 if S0_h is None else S0_h.numel() * 4
    d2h = o_h[0].numel() * 4 + S_h[0].numel() * 4
    if dstep is not None:
        h2d += sum(t.numel() * t.element_size() for t in dh.values())
        d2h += od_h[0].numel() * 4

    def dev_like(t):
        return torch.empty(t.shape, dtype=t.dtype, device=dev)

    din = [{n: dev_like(host[n]) for n in names} for _ in range(NB)]
    dcu = [dev_like(cu_h) for _ in range(NB)]
    ds0 = [None if S0_h is None else dev_like(S0_h) for _ in range(NB)]
    dout = [(torch.empty((T, H, DV), dtype=torch.float32, device=dev),
             torch.empty((N, H, DK, DV), dtype=torch.float32, device=dev)) for _ in range(NB)]
    if dstep is not None:
        ddin = [{n: dev_like(dh[n]) for n in names} for _ in range(NB)]
        dod = [torch.empty((N, H, DV), dtype=torch.float32, device=dev) for _ in range(NB)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_comp = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [torch.cuda.Event() for _ in range(NB)]
    used = [False] * NB

    def step(i):
        bsel = i % NB
        with torch.cuda.stream(s_in):
            if used[bsel]:
                s_in.wait_event(ev_comp[bsel])          # step i-2 has read these inputs
            for n in names:
                din[bsel][n].copy_(host[n], non_blocking=True)
            dcu[bsel].copy_(cu_h, non_blocking=True)
            if S0_h is not None:
                ds0[bsel].copy_(S0_h, non_blocking=True)
            if dstep is not None:
                for n in names:
                    ddin[bsel][n].copy_(dh[n], non_blocking=True)
            ev_in[bsel].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[bsel])
            if used[bsel]:
                s_comp.wait_event(ev_out[bsel])         # step i-2's outputs are read out
            d = din[bsel]
            o, S = dout[bsel]
            kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], dcu[bsel], S0=ds0[bsel],
                                chunk=pre.chunk, o=o, S_out=S)
            if dstep is not None:
                x = ddin[bsel]
                kda.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], S, o=dod[bsel])
            ev_comp[bsel].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[bsel])
            o, S = dout[bsel]
            o_h[bsel].copy_(o, non_blocking=True)
            S_h[bsel].copy_(S, non_blocking=True)
            if dstep is not None:
                od_h[bsel].copy_(dod[bsel], non_blocking=True)
            ev_out[bsel].record(s_out)
        used[bsel] = True

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(args.steps):
        step(i)
    b.record(s_out)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, ws, dev)
    tc = pre.dtype == "bf16" and pre.chunk == 64 and T > 0
    return {"value": round(job_throughput(T, ws, ms), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "copy-in / compute / copy-out streams, two buffer sets",
            "gpu_launches": ((3 if tc else 1) + (dstep is not None)) * args.steps}


def _oracle_sample(pre, heads):
    """Time the oracle on the first `heads` heads of every sequence."""
    import oracle
    units = [(n, h) for n in range(pre.N) for h in range(heads)]
    threads = min(oracle.default_threads(), len(units))
    oracle.build()
    t = time.perf_counter()
    oracle.prefill(pre, units=units, threads=threads)
    dt = time.perf_counter() - t
    return dt, threads, units


def _sample_heads(pre, args):
    # about 4e5 token-heads per sample: roughly 10-30 s of fp64 CPU work
    return max(1, min(pre.H, args.cpu_heads or int(round(4e5 / max(1, pre.T)))))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _single_core_anchor(args):
    """The oracle on one core over 16 heads of the 4K prefill: the scaling
    anchor of the multi-core numbers (tokens/s counting the sampled
    token-heads as full-width tokens)."""
    import oracle
    pre = ki.workload_prefill("prefill_4k")
    heads = 16
    units = [(0, h) for h in range(heads)]
    oracle.build()
    t = time.perf_counter()
    oracle.prefill(pre, units=units, threads=1)
    dt = time.perf_counter() - t
    return {"workload": "prefill_4k", "value": round(pre.T * heads / pre.H / dt, 2), "unit": UNIT,
            "cores": 1, "sample": "%d of %d heads (%d token-heads), %.2f s" % (heads, pre.H, pre.T * heads, dt)}


def _cpu_baseline(pre, args):
    heads = _sample_heads(pre, args)
    dt, threads, units = _oracle_sample(pre, heads)
    tokens_equiv = pre.T * heads / pre.H      # sampled token-heads as full-width tokens
    out = {"value": round(tokens_equiv / dt, 2), "unit": UNIT, "cores": threads,
           "kind": "oracle", "cpu_model": cpu_model(),
           "threads": "%d worker threads (one (sequence, head) unit each at a time; the C oracle "
                      "itself is single-threaded, OMP_NUM_THREADS=%s is not used)"
                      % (threads, os.environ.get("OMP_NUM_THREADS", "unset")),
           "host_cores": _host_cores(),
           "sample": "fp64 sequential oracle on %d of %d heads of every sequence (%d token-heads, "
                     "%.1f s); value counts the sampled token-heads as %.0f full-width tokens"
                     % (heads, pre.H, pre.T * heads, dt, tokens_equiv)}
    if not args.no_anchor:
        out["single_core_anchor"] = _single_core_anchor(args)
    return out


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    """The CPU oracle, timed as it stands on the host cores, on the same
    workload, metric and unit (bounded sample per step)."""
    ws, rank, local = _dist()
    if rank != 0:
        return
    import oracle
    wl = args.workload
    pre = ki.workload_prefill(wl) if wl != "varlen_64k" else ki.workload_varlen_with_decode(wl)[0]
    heads = _sample_heads(pre, args)
    oracle.build()
    for _ in range(args.warmup):
        _oracle_sample(pre, heads)
    t = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        _, threads, _ = _oracle_sample(pre, heads)
    dt = (time.perf_counter() - t) / args.steps
    tokens_equiv = pre.T * heads / pre.H
    value = tokens_equiv / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl, "H": pre.H, "T": pre.T, "N": pre.N, "chunk": pre.chunk,
                   "dk": DK, "dv": DV, "qkv": pre.dtype, "S0": pre.S0 is not None,
                   "lens": [int(x) for x in np.diff(pre.cu_seqlens)] if pre.N > 1 else None,
                   "then_decode": wl == "varlen_64k"},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": "%d of %d heads of every sequence per step (the prefill; "
                                   "value counts the sampled token-heads as full-width tokens)"
                                   % (heads, pre.H)},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="varlen_64k", choices=PREFILL_WORKLOADS,
                    help="headline workload (default: the largest, the 65,536-token varlen "
                         "batch then one decode step); the others run as legs")
    ap.add_argument("--no-legs", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--no-anchor", action="store_true",
                    help="skip the single-core oracle anchor of the CPU baseline")
    ap.add_argument("--cpu-heads", type=int, default=0,
                    help="heads per sequence in the oracle sample (default: ~4e5 token-heads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-layer", action="store_true",
                    help="skip the layer leg (prologue, gated prefill, fused layer decode)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end leg (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("bench.py: warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
