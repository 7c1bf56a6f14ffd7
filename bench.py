"""Benchmark of the Mamba-3 scan on B300: prefill tokens/s (headline), decode
tokens/s, roofline fractions, end-to-end and CPU-oracle baselines.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one m3_scan_fwd call on the 1.5B-layer SISO prefill workload
(batch 8, L 2048, H 32, P 64, N 128, R 1, chunk 64, bf16 activations, fp32
state). Inputs are resident in HBM; L2 is flushed (a 256 MiB write) before
every timed launch, and only the launch is timed, with CUDA events on the
launching stream. Under torchrun each rank runs its own copy of the workload
on its own GPU (independent sequences: no data-path collective), and the
aggregate is all ranks' tokens over the slowest rank's time.

Printed on rank 0: one JSON line. Besides the contract keys it carries
  roofline         HBM roof of the prefill kernel (algorithmic bytes / time)
  roofline_tensor  tensor-pipe roof of the same kernel (algorithmic FLOPs / time)
  decode           1024-step CUDA-graph decode, batch 128 x 32 heads, R = 1 and 4
  decode_tokens    multi-token decode (8 tokens per call, state read and written
                   once per call), same batch, R = 1 and 4
  prefill_mimo     the R = 4 prefill workload (chunk 16)
  prefill_chunked  the headline workload as two calls of 1024 tokens (continuation)
  prefill_backward the backward pass (all gradients) of the headline workload
  e2e              through the C ABI from pinned host buffers, copies included
  cpu_baseline     the fp64 CPU oracle on a bounded sample of the workload
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import m3synth  # noqa: E402

METRIC = "Mamba-3 scan prefill tok/s & decode tok/s per B300; % of roofline"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p["bf16_tflops_sustained"]), src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, src="fallback")


def prefill_bytes(s: m3synth.ScanShape) -> int:
    """Algorithmic HBM bytes of one prefill call: every input read once, every
    output written once (activations in bf16, dt/lambda/theta/state fp32)."""
    act = 2 if s.bf16 else 4
    b, L, H, G, P, N, R = s.batch, s.seqlen, s.heads, s.groups, s.headdim, s.dstate, s.R
    return (2 * b * L * H * P * R * act          # x in, y out
            + 2 * b * L * H * 4                  # dt, lambda
            + 2 * b * L * G * N * R * act        # B, C
            + b * L * G * (N // 2) * 4           # theta
            + b * H * N * P * 4                  # final state
            + H * 4 + 2 * H * N * R * 4)         # A, biases


def prefill_flops(s: m3synth.ScanShape) -> int:
    """Dense chunked-SSD FLOPs: per token and head 2 Q R^2 (N + P) for the
    intra-chunk block (scores and their product with X over the full Q R x Q R
    tile) plus 4 R N P for the state read-out and the chunk-state update."""
    Q, R, N, P = s.chunk, s.R, s.dstate, s.headdim
    return s.batch * s.seqlen * s.heads * (2 * Q * R * R * (N + P) + 4 * R * N * P)


def prefill_flops_causal(s: m3synth.ScanShape) -> int:
    """The same count with only the causal half of the intra-chunk block: per
    token and head Q R^2 (N + P) + 4 R N P."""
    Q, R, N, P = s.chunk, s.R, s.dstate, s.headdim
    return s.batch * s.seqlen * s.heads * (Q * R * R * (N + P) + 4 * R * N * P)


def cpu_model() -> str:
    """The host CPU's model name (for the CPU baseline's record)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def decode_bytes(s: m3synth.ScanShape, act: int = 2) -> int:
    """Per decode step: state read + write, plus the token's activations
    (``act`` bytes per activation element)."""
    b, H, G, P, N, R = s.batch, s.heads, s.groups, s.headdim, s.dstate, s.R
    return (2 * b * H * N * P * 4 + 3 * b * H * P * R * act + 3 * b * G * N * R * act
            + b * G * (N // 2) * 4 + 2 * b * H * 4)


def decode_tokens_bytes(s: m3synth.ScanShape, K: int) -> int:
    """Per multi-token call: the state read + written once, plus the K tokens'
    activations (x, out, B, C, theta, dt, lambda) and the token before the block."""
    b, H, G, P, N, R = s.batch, s.heads, s.groups, s.headdim, s.dstate, s.R
    act = 2
    per_token = (2 * b * H * P * R * act + 2 * b * G * N * R * act + b * G * (N // 2) * 4
                 + 2 * b * H * 4)
    return 2 * b * H * N * P * 4 + K * per_token + b * H * P * R * act + b * G * N * R * act


class Clocks:
    """nvidia-smi sampling during a timed region (median SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def _traffic_from_profiles(kernel_tag: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it matches the
    current kernel source (otherwise None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    src = os.path.join(ROOT, "selective_state_space_129_b300", "csrc", kernel_tag)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    sha = hashlib.sha1(open(src, "rb").read()).hexdigest()[:12]
    for line in open(path):
        if line.startswith("traffic:"):
            f = dict(kv.split("=", 1) for kv in line[len("traffic:"):].split())
            if f.get("source") == kernel_tag and f.get("sha") == sha:
                return int(f["bytes_per_launch"])
    return None


# ---------------------------------------------------------------- oracle arm
def _stack_heads(shape, inp, bs, hs):
    """k single-head sequences of the workload stacked along the batch axis."""
    g = hs // (shape.heads // shape.groups)
    k = len(bs)
    sl = lambda a, ix: np.stack([a[bs[i], :, ix[i]] for i in range(k)])[:, :, None]
    h0 = int(hs[0])
    return dict(x=sl(inp["x"], hs), dt=sl(inp["dt"], hs), A=inp["A"][h0:h0 + 1],
                lam=sl(inp["lam"], hs), B=sl(inp["B"], g), C=sl(inp["C"], g),
                theta=sl(inp["theta"], g), B_bias=inp["B_bias"][h0:h0 + 1],
                C_bias=inp["C_bias"][h0:h0 + 1])


def oracle_rate(shape, inp, budget_s=12.0):
    """Oracle tok/s on whole single-head sequences of the workload (OpenMP over
    the stacked sequences, all host cores), sized to about ``budget_s``."""
    from oracle import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(7)

    def timed(k):
        sub = _stack_heads(shape, inp, rng.integers(0, shape.batch, k),
                           rng.integers(0, shape.heads, k))
        t0 = time.perf_counter()
        oracle.scan_seq(nthreads=threads, **sub)
        return k * shape.seqlen, time.perf_counter() - t0

    k0 = min(threads, 16)
    tok, el = timed(k0)
    k = int(max(k0, min(256, k0 * budget_s / max(el, 1e-6))))
    k = max(threads, (k // threads) * threads) if k >= threads else k
    tok, el = timed(k)
    sample = ("%d whole single-head sequences of %d tokens drawn from the workload "
              "(timing sample; A and biases of one head)" % (k, shape.seqlen))
    return tok / el, min(threads, k), sample


# ---------------------------------------------------------------- ranks
# One process per GPU, each on its own batch (independent replicas, weak
# scaling): no data-path collective, only the barrier around the timed region
# and the max over ranks of the measured time.
def rank_seed(idx, rank):
    """Input seed of a rank: the workload's seed for rank 0, distinct per rank."""
    return idx + 1000 * rank


def max_over_ranks(torch, value, world, device):
    """The largest value over all ranks (every rank gets it); value itself at N = 1."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_per_rank, world, ms):
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return tokens_per_rank * world / (ms * 1e-3)


def headline_config(shape, world, name="prefill_siso"):
    """A prefill workload's config (the headline's is identical in both arms)."""
    return {"workload": "%s b%d L%d H%d P%d N%d G%d R%d chunk%d" % (
                name, shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate,
                shape.groups, shape.R, shape.chunk),
            "global_batch": shape.batch * world, "seq_len": shape.seqlen,
            "parallelism": "independent replicas" if world > 1 else "single GPU",
            "l2": "flushed before every timed launch (256 MiB write)",
            "state": "fp32", "activations": "bf16"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle timed as it stands on the host cores."""
    if rank != 0:
        return
    idx, shape = m3synth.WORKLOADS["prefill_siso"]
    inp = m3synth.scan_inputs(shape, seed=idx)
    from oracle import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(17)
    k = min(shape.batch * shape.heads, max(threads, 8))

    def step():
        sub = _stack_heads(shape, inp, rng.integers(0, shape.batch, k),
                           rng.integers(0, shape.heads, k))
        oracle.scan_seq(nthreads=threads, **sub)
        return k * shape.seqlen

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    tok = sum(step() for _ in range(args.steps))
    el = time.perf_counter() - t0
    value = tok / el
    sample = "%d whole sequences of %d tokens per step (one head each)" % (k, shape.seqlen)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(shape, world),
        "note": "fp64 CPU oracle (sequential explicit-rotation recurrence) on the host cores",
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def to_device(inp, bf16, dev):
    """Seeded numpy inputs -> torch tensors (activations bf16 when asked)."""
    import torch
    out = {}
    for k, v in inp.items():
        if k == "bits":
            continue
        t = torch.from_numpy(np.ascontiguousarray(v))
        if bf16 and k in ("x", "B", "C"):
            t = t.to(torch.bfloat16)
        out[k] = t.to(dev)
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import selective_state_space_129_b300 as m3

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    m3.load()
    peaks = _peaks()
    stream = torch.cuda.current_stream()

    if args.only in ("decode_siso", "decode_mimo"):
        if rank == 0:
            print(json.dumps(bench_decode(torch, m3, dev, args.only, peaks,
                                          steps=args.decode_steps)), flush=True)
        return
    if args.only in ("decode_tokens_siso", "decode_tokens_mimo"):
        if rank == 0:
            name = args.only.replace("tokens_", "")
            print(json.dumps(bench_decode_tokens(torch, m3, dev, name, peaks,
                                                 calls=args.decode_steps)), flush=True)
        return
    if args.only == "prefill_backward":
        if rank == 0:
            print(json.dumps(bench_backward(torch, m3, dev)), flush=True)
        return
    if args.only == "prefill_long":
        if rank == 0:
            print(json.dumps(bench_prefill_long(torch, m3, dev, args, peaks)), flush=True)
        return
    if args.only == "prefill_bcnorm":
        if rank == 0:
            print(json.dumps({k: bench_prefill_other(torch, m3, dev, w, args, peaks, bc_norm=True)
                              for k, w in (("siso", "prefill_siso"),
                                           ("mimo_r4", "prefill_mimo"))}), flush=True)
        return
    if args.only == "fp32_mode":
        if rank == 0:
            print(json.dumps({
                "prefill_siso": bench_prefill_other(torch, m3, dev, "prefill_siso", args, peaks,
                                                    fp32=True),
                "decode_siso": bench_decode(torch, m3, dev, "decode_siso", peaks, fp32=True),
                "decode_mimo_r4": bench_decode(torch, m3, dev, "decode_mimo", peaks,
                                               fp32=True)}), flush=True)
        return
    name = args.only if args.only in ("prefill_siso", "prefill_mimo") else "prefill_siso"
    idx, shape = m3synth.WORKLOADS[name]
    inp = m3synth.scan_inputs(shape, seed=rank_seed(idx, rank))
    d = to_device(inp, True, dev)
    out = torch.empty_like(d["x"])
    fs = torch.empty((shape.batch, shape.heads, shape.dstate, shape.headdim),
                     dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def launch():
        m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"], R=shape.R,
                       chunk=shape.chunk, out=out, final_state=fs, B_bias=d["B_bias"],
                       C_bias=d["C_bias"], stream=stream)

    # the clock sampler starts before the warm-up, so that its start-up pause
    # does not leave an idle (down-clocked) GPU right before the timed steps
    with Clocks(local_rank) as clk:
        for _ in range(args.warmup):
            flush.zero_()
            launch()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            launch()
            e1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    status = m3.m3_device_status()
    times = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms = sum(times) / len(times)
    ms = max_over_ranks(torch, ms, world, dev)
    value = job_rate(shape.tokens, world, ms)
    del flush
    torch.cuda.empty_cache()
    # end to end through the public call, on every rank at once (whole-job rate)
    e2e = bench_e2e(torch, m3, dev, shape, inp, args, world) if args.only == "all" else None
    if rank != 0:
        return

    nbytes = prefill_bytes(shape)
    nflops = prefill_flops(shape)
    gbs = nbytes / (ms * 1e-3) / 1e9
    tfs = nflops / (ms * 1e-3) / 1e12
    tc_kernel = "scan_tc.cu"
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(shape, world, name),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm"], "traffic": _traffic_from_profiles(tc_kernel),
                     "algorithmic_bytes": nbytes, "peak_source": peaks["src"] + " (burst)"},
        "roofline_tensor": {"bound": "tensor", "achieved": tfs, "peak": peaks["bf16"],
                            "unit": "TFLOP/s", "frac": tfs / peaks["bf16"],
                            "algorithmic_flops": nflops,
                            "frac_causal_half": prefill_flops_causal(shape) / (ms * 1e-3) / 1e12
                                                / peaks["bf16"],
                            "algorithmic_flops_causal_half": prefill_flops_causal(shape),
                            "peak_source": peaks["src"] + " bf16 dense (burst)"},
        "clocks": clk.summary(),
        "gpu_launches": args.steps,
        "device_status": m3.m3_status_string(status),
    }
    if args.only != "all":
        # a single workload (used for profiling): no side benchmarks
        print(json.dumps(line), flush=True)
        return
    line["prefill_mimo"] = bench_prefill_other(torch, m3, dev, "prefill_mimo", args, peaks)
    line["prefill_bcnorm"] = {
        "siso": bench_prefill_other(torch, m3, dev, "prefill_siso", args, peaks, bc_norm=True),
        "mimo_r4": bench_prefill_other(torch, m3, dev, "prefill_mimo", args, peaks,
                                       bc_norm=True)}
    line["fp32_mode"] = {
        "prefill_siso": bench_prefill_other(torch, m3, dev, "prefill_siso", args, peaks,
                                            fp32=True),
        "decode_siso": bench_decode(torch, m3, dev, "decode_siso", peaks, fp32=True),
        "decode_mimo_r4": bench_decode(torch, m3, dev, "decode_mimo", peaks, fp32=True)}
    line["prefill_chunked"] = bench_prefill_chunked(torch, m3, dev, args)
    line["prefill_backward"] = bench_backward(torch, m3, dev)
    line["prefill_backward"]["over_forward"] = line["prefill_backward"]["ms"] / ms
    line["prefill_long"] = bench_prefill_long(torch, m3, dev, args, peaks)
    line["decode"] = {"siso": bench_decode(torch, m3, dev, "decode_siso", peaks),
                      "mimo_r4": bench_decode(torch, m3, dev, "decode_mimo", peaks)}
    sis, mim = line["decode"]["siso"], line["decode"]["mimo_r4"]
    if sis.get("ms_per_step") and mim.get("ms_per_step"):
        line["decode"]["r4_over_r1_latency"] = mim["ms_per_step"] / sis["ms_per_step"]
    line["decode_tokens"] = {
        "siso_k%d" % DECODE_BLOCK: bench_decode_tokens(torch, m3, dev, "decode_siso", peaks),
        "mimo_r4_k%d" % DECODE_BLOCK: bench_decode_tokens(torch, m3, dev, "decode_mimo", peaks)}
    line["e2e"] = e2e
    if not args.no_cpu_baseline:
        rate, cores, sample = oracle_rate(shape, inp)
        line["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": cores,
                                "kind": "oracle", "sample": sample, "cpu_model": cpu_model()}
    print(json.dumps(line), flush=True)


def bench_prefill_other(torch, m3, dev, name, args, peaks, bc_norm=False, fp32=False):
    """One prefill workload timed like the headline. ``bc_norm``: B and C are
    un-normalised (the recipe's vectors times a seeded per-vector scale) and
    the call fuses BCNorm (M3_FLAG_BC_NORM). ``fp32``: fp32 activations, the
    fp32 precision mode (CUDA-core kernel)."""
    idx, shape = m3synth.WORKLOADS[name]
    if fp32:
        shape = dataclasses.replace(shape, bf16=False)
    inp = m3synth.scan_inputs(shape, seed=idx)
    if bc_norm:
        rng = np.random.default_rng(idx)
        for k in ("B", "C"):
            v = inp[k]
            sc = rng.uniform(0.05, 20.0, size=v.shape[:3] + (1,) + v.shape[4:]).astype(np.float32)
            inp[k] = m3synth.to_bf16(v * sc)
    d = to_device(inp, not fp32, dev)
    out = torch.empty_like(d["x"])
    fs = torch.empty((shape.batch, shape.heads, shape.dstate, shape.headdim),
                     dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def launch():
        m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"], R=shape.R,
                       chunk=shape.chunk, out=out, final_state=fs, B_bias=d["B_bias"],
                       C_bias=d["C_bias"], stream=stream, bc_norm=bc_norm)

    steps = min(args.steps, 5) if fp32 else args.steps
    for _ in range(args.warmup):
        flush.zero_()
        launch()
    times = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = sum(times) / len(times)
    nbytes, nflops = prefill_bytes(shape), prefill_flops(shape)
    r = {"workload": "%s b%d L%d H%d P%d N%d R%d chunk%d%s%s" % (
             name, shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate,
             shape.R, shape.chunk, ", fp32 activations" if fp32 else "",
             ", un-normalised B/C with BCNorm fused" if bc_norm else ""),
         "tok_s": shape.tokens / (ms * 1e-3), "ms": ms,
         "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm"]}
    r["tensor_frac"] = nflops / (ms * 1e-3) / 1e12 / peaks["bf16"]
    if fp32:
        # the fp32 mode runs on the tensor cores with split fp16 operands (three
        # MMAs per product): tensor_frac counts the algorithm's FLOPs once
        r["kernel"] = ("tensor cores, fp32 activations as fp16 high + residual tiles, "
                       "three products per contraction")
        r["tensor_issued_frac"] = 3 * r["tensor_frac"]
    return r


def bench_prefill_chunked(torch, m3, dev, args, pieces=2):
    """The headline prefill workload run as ``pieces`` consecutive calls (the
    first m3_scan_fwd, the others m3_scan_fwd_state continuing from the state
    and last token of the call before), timed like the single call."""
    idx, shape = m3synth.WORKLOADS["prefill_siso"]
    inp = m3synth.scan_inputs(shape, seed=idx)
    d = to_device(inp, True, dev)
    Lp = shape.seqlen // pieces
    seq = ("x", "dt", "lam", "B", "C", "theta")
    parts = [{k: (v[:, i * Lp:(i + 1) * Lp].contiguous() if k in seq else v) for k, v in d.items()}
             for i in range(pieces)]
    prevs = [None] + [{"B": parts[i]["B"][:, -1].contiguous(), "x": parts[i]["x"][:, -1].contiguous()}
                      for i in range(pieces - 1)]
    outs = [torch.empty_like(p["x"]) for p in parts]
    st = torch.empty((shape.batch, shape.heads, shape.dstate, shape.headdim),
                     dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def launch():
        for i, (p, pv) in enumerate(zip(parts, prevs)):
            if i == 0:
                m3.m3_scan_fwd(p["x"], p["dt"], p["A"], p["lam"], p["B"], p["C"], p["theta"],
                               R=shape.R, chunk=shape.chunk, out=outs[i], final_state=st,
                               B_bias=p["B_bias"], C_bias=p["C_bias"], stream=stream)
            else:
                m3.m3_scan_fwd_state(p["x"], p["dt"], p["A"], p["lam"], p["B"], p["C"],
                                     p["theta"], R=shape.R, chunk=shape.chunk, state=st,
                                     B_prev=pv["B"], x_prev=pv["x"], out=outs[i],
                                     B_bias=p["B_bias"], C_bias=p["C_bias"], stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        launch()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = sum(times) / len(times)
    return {"workload": "prefill_siso b%d L%d as %d calls of %d tokens (m3_scan_fwd, then "
                        "m3_scan_fwd_state)" % (shape.batch, shape.seqlen, pieces, Lp),
            "tok_s": shape.tokens / (ms * 1e-3), "ms": ms, "gpu_launches": pieces + pieces - 1}


def bench_backward(torch, m3, dev, reps=3):
    """m3_scan_bwd on the headline prefill workload (gradients of <y, dy> +
    <h_final, d_final>), timed like the forward call (L2 flushed first)."""
    idx, shape = m3synth.WORKLOADS["prefill_siso"]
    inp = m3synth.scan_inputs(shape, seed=idx)
    d = to_device(inp, True, dev)
    gen = torch.Generator(device=dev).manual_seed(idx)
    dy = torch.randn(d["x"].shape, device=dev, generator=gen).to(torch.bfloat16)
    dfin = torch.randn((shape.batch, shape.heads, shape.dstate, shape.headdim), device=dev,
                       generator=gen)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    # the scratch a training loop allocates once and passes to every call
    dims = m3.make_dims(shape.batch, shape.seqlen, shape.heads, shape.groups, shape.headdim,
                        shape.dstate, m3.M3_BF16)
    ws_bytes = m3.m3_scan_bwd_workspace_bytes(dims, shape.R)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)

    def launch():
        m3.m3_scan_bwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"], dy,
                       R=shape.R, d_final=dfin, B_bias=d["B_bias"], C_bias=d["C_bias"],
                       stream=stream, workspace=ws)

    launch()
    times = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = sum(times) / len(times)
    return {"workload": "prefill_siso b%d L%d H%d P%d N%d R%d, backward (all gradients)" % (
                shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate, shape.R),
            "tok_s": shape.tokens / (ms * 1e-3), "ms": ms, "workspace_bytes": ws_bytes,
            "kernel": "chunked on the tensor cores (mma.sync TF32): chunk contributions, "
                      "boundary-state scans, per-chunk gradients"}


def device_inputs(torch, shape, dev, seed):
    """The synthetic recipe's distributions drawn directly on the device (torch
    RNG): timing inputs for the long-context workloads, whose host-side
    generation would dominate the run. Parity tests use m3synth's seeded
    numpy inputs."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    b, L, H, G, P, N, R = (shape.batch, shape.seqlen, shape.heads, shape.groups, shape.headdim,
                           shape.dstate, shape.R)
    f32 = dict(device=dev, dtype=torch.float32)

    def rn(*sz):
        return torch.randn(*sz, generator=gen, **f32)

    def bc():
        v = rn(b, L, G, N, R)
        v = v / torch.sqrt(v.square().mean(dim=-2, keepdim=True) + 1e-6)
        return v.to(torch.bfloat16)

    A = -torch.exp(torch.rand(H, generator=gen, **f32) * float(np.log(16.0)))
    dt = torch.nn.functional.softplus(rn(b, L, H) * 0.5 - 1.0)
    lam = torch.sigmoid(rn(b, L, H))
    theta = (torch.rand(b, L, G, N // 2, generator=gen, **f32) * 2.0 - 1.0) * float(np.pi)
    return dict(A=A, dt=dt, lam=lam, theta=theta, B=bc(), C=bc(), B_bias=0.1 * rn(H, N, R),
                C_bias=0.1 * rn(H, N, R), x=rn(b, L, H, P, R).to(torch.bfloat16))


def bench_prefill_long(torch, m3, dev, args, peaks):
    """The long-context workloads (b1 L65536 H32 P64): SISO N64 and N128 (chunk
    64), MIMO R4 N128 (chunk 16). 32 sequences for 148 SMs: the scan runs
    segmented (state-only pass, combine, full pass)."""
    res = {}
    stream = torch.cuda.current_stream()
    for name in ("long_siso_n64", "long_siso_n128", "long_mimo_n128"):
        idx, shape = m3synth.WORKLOADS[name]
        d = device_inputs(torch, shape, dev, seed=idx)
        out = torch.empty_like(d["x"])
        fs = torch.empty((shape.batch, shape.heads, shape.dstate, shape.headdim),
                         dtype=torch.float32, device=dev)
        dims = m3.make_dims(shape.batch, shape.seqlen, shape.heads, shape.groups, shape.headdim,
                            shape.dstate, m3.M3_BF16)
        ws_bytes = m3.m3_scan_workspace_bytes(dims, shape.R, shape.chunk)
        ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)

        def launch():
            m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["lam"], d["B"], d["C"], d["theta"],
                           R=shape.R, chunk=shape.chunk, out=out, final_state=fs,
                           B_bias=d["B_bias"], C_bias=d["C_bias"], workspace=ws, stream=stream)

        for _ in range(3):
            launch()
        times = []
        for _ in range(max(3, min(args.steps, 5))):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = sum(times) / len(times)
        nbytes, nflops = prefill_bytes(shape), prefill_flops(shape)
        res[name] = {"workload": "%s b%d L%d H%d P%d N%d R%d chunk%d" % (
                         name, shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate,
                         shape.R, shape.chunk),
                     "tok_s": shape.tokens / (ms * 1e-3), "ms": ms,
                     "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm"],
                     "tensor_frac": nflops / (ms * 1e-3) / 1e12 / peaks["bf16"],
                     "workspace_bytes": ws_bytes,
                     "inputs": "recipe distributions drawn on the device (torch RNG)"}
        # the most the tensor pipe could be busy with the scan at the HBM
        # roof: algorithmic FLOPs over the time the algorithmic bytes take
        ceil = (nflops / 1e12 / peaks["bf16"]) / (nbytes / 1e9 / peaks["hbm"])
        res[name]["tensor_frac_ceiling_at_hbm_roof"] = ceil
        if ceil < 0.5:
            res[name]["note"] = ("a 50%% tensor target is out of reach at this shape: even at "
                                 "the HBM roof the tensor pipe could be at most %.0f%% busy"
                                 % (100 * ceil))
        del d, out, fs, ws
        torch.cuda.empty_cache()
    return res


def bench_decode(torch, m3, dev, name, peaks, n_sets=16, steps=m3synth.DECODE_STEPS,
                 fp32=False):
    """1024 decode steps captured in one CUDA graph; per-step inputs cycle over
    ``n_sets`` seeded token sets (B_prev/x_prev are the previous set's).
    ``fp32``: fp32 activations (the fp32 precision mode)."""
    idx, shape = m3synth.WORKLOADS[name]
    if fp32:
        shape = dataclasses.replace(shape, bf16=False)
    sets = [to_device(m3synth.decode_inputs(shape, seed=idx, step=i), not fp32, dev)
            for i in range(n_sets)]
    st = torch.zeros((shape.batch, shape.heads, shape.dstate, shape.headdim),
                     dtype=torch.float32, device=dev)
    out = torch.empty_like(sets[0]["x"])
    s = torch.cuda.Stream(device=dev)

    def step(i, stream):
        cur, prev = sets[i % n_sets], sets[(i - 1) % n_sets]
        m3.m3_decode_step(st, cur["x"], cur["dt"], cur["A"], cur["lam"], cur["B"], cur["C"],
                          cur["theta"], R=shape.R, B_prev=prev["B"], x_prev=prev["x"], out=out,
                          B_bias=cur["B_bias"], C_bias=cur["C_bias"], stream=stream)

    with torch.cuda.stream(s):
        for i in range(8):
            step(i, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            step(i, s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / (reps * steps)
    nbytes = decode_bytes(shape, 4 if fp32 else 2)
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    return {"workload": "%s b%d H%d P%d N%d R%d, %d steps in one CUDA graph%s" % (
                name, shape.batch, shape.heads, shape.headdim, shape.dstate, shape.R, steps,
                ", fp32 activations" if fp32 else ""),
            "tok_s": shape.batch / (ms_step * 1e-3), "ms_per_step": ms_step,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "algorithmic_bytes": nbytes},
            "gpu_launches": steps * reps,
            "l2": "state 134 MB exceeds the 126 MB L2; no flush between steps"}


DECODE_BLOCK = 8  # tokens per multi-token decode call
# fp32 CUDA-core peak: 148 SMs x 128 FMA lanes x 2 flop x 2.032 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def bench_decode_tokens(torch, m3, dev, name, peaks, K=DECODE_BLOCK, calls=128, n_sets=4):
    """Multi-token decode: ``calls`` calls of K tokens each for the 128 x 32
    decode batch, captured in one CUDA graph; the blocks cycle over ``n_sets``
    seeded K-token sets (each block's B_prev / x_prev are the last token of
    the block before). tok/s = 128 K calls / time."""
    idx, base = m3synth.WORKLOADS[name]
    shape = m3synth.ScanShape(base.batch, K, base.heads, base.groups, base.headdim, base.dstate,
                              R=base.R, chunk=1)
    raw = [m3synth.scan_inputs(shape, seed=100 * idx + i) for i in range(n_sets)]
    for r in raw[1:]:  # one head's A and biases for the whole run
        r["A"], r["B_bias"], r["C_bias"] = raw[0]["A"], raw[0]["B_bias"], raw[0]["C_bias"]
    sets = [to_device(r, True, dev) for r in raw]
    last = [{"B": s["B"][:, K - 1].contiguous(), "x": s["x"][:, K - 1].contiguous()} for s in sets]
    st = torch.zeros((shape.batch, shape.heads, shape.dstate, shape.headdim),
                     dtype=torch.float32, device=dev)
    out = torch.empty_like(sets[0]["x"])
    s = torch.cuda.Stream(device=dev)

    def call(i, stream):
        cur, prev = sets[i % n_sets], last[(i - 1) % n_sets]
        m3.m3_decode_tokens(st, cur["x"], cur["dt"], cur["A"], cur["lam"], cur["B"], cur["C"],
                            cur["theta"], R=shape.R, B_prev=prev["B"], x_prev=prev["x"],
                            out=out, B_bias=cur["B_bias"], C_bias=cur["C_bias"], stream=stream)

    with torch.cuda.stream(s):
        for i in range(4):
            call(i, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(calls):
            call(i, s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    ms_call = e0.elapsed_time(e1) / (reps * calls)
    nbytes = decode_tokens_bytes(shape, K)
    gbs = nbytes / (ms_call * 1e-3) / 1e9
    # per state element and token: alpha Rot h (2 FMA), U (x_prev | x)^T (2R FMA), y (R FMA)
    flops = (shape.batch * shape.heads * shape.dstate * shape.headdim * K * (4 + 6 * shape.R))
    tfl = flops / (ms_call * 1e-3) / 1e12
    return {"workload": "%s b%d H%d P%d N%d R%d, %d tokens per call, %d calls in one CUDA graph"
                        % (name, shape.batch, shape.heads, shape.headdim, shape.dstate, shape.R,
                           K, calls),
            "tok_s": shape.batch * K / (ms_call * 1e-3), "ms_per_call": ms_call,
            "ms_per_token_step": ms_call / K,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "algorithmic_bytes": nbytes},
            "roofline_alu": {"bound": "alu", "achieved": tfl, "peak": FP32_PEAK_TFLOPS,
                             "unit": "TFLOP/s", "frac": tfl / FP32_PEAK_TFLOPS,
                             "algorithmic_flops": flops,
                             "peak_source": "148 SMs x 128 fp32 FMA lanes x 2 x 2.032 GHz"},
            "gpu_launches": calls * reps}


def bench_e2e(torch, m3, dev, shape, inp, args, world=1):
    """Same workload through the public call from pinned host buffers: every
    step copies its inputs host->device, runs the scan and reads its outputs
    (y and final state) back into pinned host memory. Steps are pipelined the
    way a serving loop would run them: two device buffer sets, one stream each
    for the copy in, the scan and the copy out, so that step k's scan overlaps
    step k+1's copy in and step k-1's copy out (PCIe carries both directions at
    once). All ranks run it at once; the rate is all ranks' tokens over the
    slowest rank's time."""
    host = {k: v.pin_memory() for k, v in to_device(inp, True, "cpu").items()}
    nbuf = 2
    devb = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(nbuf)]
    out = [torch.empty_like(devb[0]["x"]) for _ in range(nbuf)]
    fs = [torch.empty((shape.batch, shape.heads, shape.dstate, shape.headdim),
                      dtype=torch.float32, device=dev) for _ in range(nbuf)]
    out_h = [torch.empty_like(host["x"]).pin_memory() for _ in range(nbuf)]
    fs_h = [torch.empty(fs[0].shape, dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    in_done = [ev() for _ in range(nbuf)]
    run_done = [ev() for _ in range(nbuf)]
    out_done = [ev() for _ in range(nbuf)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + fs_h[0].numel() * 4

    def step(k):
        j = k % nbuf
        s_in.wait_event(run_done[j])    # step k - 2's scan has read buffer set j
        with torch.cuda.stream(s_in):
            for name in host:
                devb[j][name].copy_(host[name], non_blocking=True)
            in_done[j].record(s_in)
        s_run.wait_event(in_done[j])
        s_run.wait_event(out_done[j])   # step k - 2's outputs have left buffer set j
        m3.m3_scan_fwd(devb[j]["x"], devb[j]["dt"], devb[j]["A"], devb[j]["lam"], devb[j]["B"],
                       devb[j]["C"], devb[j]["theta"], R=shape.R, chunk=shape.chunk, out=out[j],
                       final_state=fs[j], B_bias=devb[j]["B_bias"], C_bias=devb[j]["C_bias"],
                       stream=s_run)
        run_done[j].record(s_run)
        s_out.wait_event(run_done[j])
        with torch.cuda.stream(s_out):
            out_h[j].copy_(out[j], non_blocking=True)
            fs_h[j].copy_(fs[j], non_blocking=True)
            out_done[j].record(s_out)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_run.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(args.steps):
        step(k)
    s_in.wait_event(out_done[(args.steps - 1) % nbuf])
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = max_over_ranks(torch, e0.elapsed_time(e1) / args.steps, world, dev)
    return {"value": job_rate(shape.tokens, world, ms), "unit": "tok/s",
            "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
            "ms_per_step": ms, "pipelined": "copy in, scan, copy out on three streams, "
                                            "two buffer sets"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="all",
                    choices=["all", "prefill_siso", "prefill_mimo", "decode_siso", "decode_mimo",
                             "decode_tokens_siso", "decode_tokens_mimo", "prefill_long",
                             "prefill_backward", "prefill_bcnorm", "fp32_mode"],
                    help="run one workload alone (profiling); the default runs them all")
    ap.add_argument("--decode-steps", type=int, default=m3synth.DECODE_STEPS,
                    help="decode steps (or multi-token calls) per CUDA graph with --only decode_*")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
