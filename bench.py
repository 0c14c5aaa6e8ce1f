#!/usr/bin/env python
"""Benchmark: effective attention TFLOPS on GB300 with quantization included.

One step = the whole hot path on one batch of seeded synthetic input already
resident in HBM: one sage_quantize_qkv call (Q and K to INT8 codes with their
block scales, V's channel maxima, then the V encode to FP8 E4M3; with K or Q
smoothing the separate quantize calls it needs) and one attention call (BF16 O
+ FP32 LSE), each replayed from a CUDA graph. Effective TFLOPS =
4*B*H*Nq*Nk*D / (summed step time). Between steps, outside the timed events,
L2 is flushed by reading a 256 MiB buffer. The default workload is the
65520-token long-video self-attention. `e2e` times the same work through
sage_attention_host: Q/K/V in page-locked host memory, O/LSE written back to
host memory, the library's pipelined copies inside the timed region. Prints
one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: the path has no exchange step); value = units of all
ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective attention TFLOPS at 1 GB300 (incl. quant) and % of dense INT8/FP8 peak"
DEFAULT_WORKLOAD = "long_video"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): fp8 4.5, fp4 13.5.
_FP8_RATIO, _FP4_RATIO = 2.0, 6.0
# Hardware exp2 (MUFU) throughput per SM per clock, measured on GB300 with a
# microbenchmark of back-to-back ex2.approx.ftz.f32.
_EX2_PER_CLK_SM = 32
# Dense tcgen05 MMA throughput per SM per clock measured on GB300 with
# microbenchmarks (M128, N >= 128, operands in shared memory): kind::f16,
# kind::f8f6f4 (E4M3) and kind::mxf4.block_scale.
_MMA_FLOP_PER_CLK_SM = {"f16": 8192.0, "f8": 16384.0, "f4": 32768.0}
_SMS = 152


def _clock_peak(fmt: int, mhz: float) -> float:
    """The attention's tensor roofline (TFLOP/s) rebuilt from the measured
    per-clock MMA rates at SM clock `mhz`: Q K^T on the f16 (INT8 codes), f4
    (MXFP4) or f8 (FP8) kind, P V on f8 (f4 for MXFP4 P V), harmonic."""
    r = _MMA_FLOP_PER_CLK_SM
    qk = {0: r["f16"], 1: r["f4"], 2: r["f8"], 3: r["f4"], 4: r["f4"]}[fmt]
    pv = r["f4"] if fmt == 4 else r["f8"]
    return 2.0 / (1.0 / qk + 1.0 / pv) * _SMS * mhz * 1e6 / 1e12


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself on one rank. Collective over the default process group."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_rank: float, steps: int, ms_max: float, world: int) -> float:
    """Whole-job TFLOP/s of `world` replicas that each ran `steps` steps of
    `flops_per_rank` work, the slowest taking `ms_max` milliseconds in total."""
    return world * flops_per_rank * steps / (ms_max * 1e-3) / 1e12


def _roofline_peak(p16: float, fmt: int) -> float:
    """Tensor roofline of the attention: half the flops (Q K^T) on the 16-bit
    pipe (INT8 codes held as FP16), the FP4 pipe (MXFP4) or the FP8 pipe (FP8
    Q/K), half (P V) on the FP8 pipe; the two halves run back to back, so the
    rates combine harmonically."""
    p_qk = p16 * {0: 1.0, 1: _FP4_RATIO, 2: _FP8_RATIO, 3: _FP4_RATIO, 4: _FP4_RATIO}[fmt]
    p_pv = p16 * (_FP4_RATIO if fmt == 4 else _FP8_RATIO)
    return 2.0 / (1.0 / p_qk + 1.0 / p_pv)


def _kernel_sources_sha256() -> str:
    """Hash of the sources that define the attention kernel, to tell whether
    committed profiler counters still describe it."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_attention_diffusion_sage_gb300", "csrc")
    for name in ("attention.cu", "attention.cuh", "sm103_ptx.cuh", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
    `kernel` on `workload` from the committed profile summaries, if they were
    taken on the current kernel sources; else None. A summary states it on a
    line `traffic: kernel=<name> workload=<name> sources_sha256=<hex>
    dram_bytes_per_launch=<int>`."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = _kernel_sources_sha256()
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                line = line.strip().strip("`")
                if not line.startswith("traffic:"):
                    continue
                kv = dict(tok.split("=", 1) for tok in line[len("traffic:"):].split() if "=" in tok)
                if (kv.get("kernel") == kernel and kv.get("workload") == workload
                        and kv.get("sources_sha256") == sha):
                    try:
                        return int(kv["dram_bytes_per_launch"])
                    except (KeyError, ValueError):
                        return None
    return None


def _quant_bytes(w, Nqp: int, Nkp: int) -> float:
    """Bytes the quantization step moves: Q and K read once (BF16) and written
    as codes (FP16-held INT8, or packed E2M1 plus one E8M0 byte per 32), V read
    by both passes (channel maxima, then encoding) and written as FP8."""
    B, H, D = w.B, w.H, w.D
    code = {0: 2.0, 1: 0.5 + 1.0 / 32, 2: 1.0, 3: 0.5 + 1.0 / 32, 4: 0.5 + 1.0 / 32}[w.fmt]
    qk = (B * w.Nq * H * D * 2 + B * H * Nqp * D * code + B * w.Nk * H * D * 2
          + B * H * Nkp * D * code)
    if w.smooth_k:  # K also read by the channel-maximum and the fixed-point-sum passes
        qk += 2 * B * w.Nk * H * D * 2
    if w.smooth_q:  # dS: K codes read, one FP32 per (query block, key) written
        qk += B * H * Nkp * D * code + B * H * (Nqp // 128) * Nkp * 4
    if w.fmt == 4:  # MXFP4 V: one pass, read once, packed E2M1 + E8M0 per 32 tokens
        return qk + B * w.Nk * H * D * 2 + B * H * D * Nkp * (0.5 + 1.0 / 32)
    return qk + B * w.Nk * H * D * 2 * 2 + B * H * D * Nkp


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"sage_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.gpu_id], stdout=self.fh, stderr=subprocess.DEVNULL)
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
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _cpu_oracle_sample(w, seconds: float, qkv, seed_rows: int = 64, nthreads: int = 0):
    """Time the CPU oracle (as it stands) on a bounded sample of workload w
    (host tensors `qkv`): quantization of the first `nh` heads' Q/K/V plus
    attention for `n` query rows of those heads, sized from a short
    calibration run to take about `seconds`. Returns (flops, time_s,
    description, rows)."""
    import numpy as np
    import oracle
    from precision_attention_diffusion_sage_gb300.inputs import bf16_bits

    q, k, v = qkv
    lens = None if w.k_lens is None else w.k_lens

    def run(nh, rows):
        qb, kb, vb = (bf16_bits(t[:, :, :nh]) for t in (q, k, v))
        t0 = time.perf_counter()
        quant_qk = {0: oracle.quantize_int8, 1: oracle.quantize_mxfp4, 2: oracle.quantize_fp8_qk,
                    3: oracle.quantize_mxfp4_hadamard, 4: oracle.quantize_mxfp4}[w.fmt]
        qm = km = ds = None
        if w.smooth_q:
            *qz, qm = oracle.quantize_int8_qsmooth(qb)
        else:
            qz = quant_qk(qb)
        if w.smooth_k:
            *kz, km = oracle.quantize_int8_smooth(kb, lens=lens)
        else:
            kz = quant_qk(kb, lens=lens)
        vz = (oracle.quantize_v_mxfp4(vb, lens=lens) if w.fmt == 4
              else oracle.quantize_v_fp8(vb, lens=lens))
        if w.smooth_q:
            ds = oracle.delta_s(kz[0], kz[1], qm, Nq=w.Nq, Nk=w.Nk, k_mean=km)
        # rotated MXFP4: MXFP4 codes of QH and KH, logits (QH)(KH)^T / 128
        afmt, c = (1, 1.0 / math.sqrt(w.D) / 128) if w.fmt == 3 else (w.fmt, None)
        oracle.attention(afmt, *qz, *kz, *vz, Nq=w.Nq, Nk=w.Nk, k_lens=lens, rows=rows,
                         softmax_scale=c, nthreads=nthreads, k_mean=km, delta_s=ds)
        return time.perf_counter() - t0

    def rows_of(n):
        return np.linspace(0, w.Nq - 1, n).astype(np.int64)

    t_cal = run(1, rows_of(min(seed_rows, w.Nq)))
    units = min(seed_rows, w.Nq) * seconds / max(t_cal, 1e-3)   # (head, row) pairs
    if units <= w.Nq:
        nh, n = 1, int(max(min(seed_rows, w.Nq), units))
    else:
        nh, n = int(min(w.H, math.ceil(units / w.Nq))), w.Nq
    dt = run(nh, rows_of(n))
    nk_sum = sum(w.k_lens) if w.k_lens else w.B * w.Nk
    flops = 4.0 * nh * n * nk_sum * w.D
    desc = (f"oracle on heads 0..{nh - 1} of every batch: full Q/K/V quantization of those heads "
            f"+ attention for {n} of {w.Nq} query rows each")
    return flops, dt, desc, n


def run_reference(args, w):
    """The CPU oracle as the reference arm, on this run's workload and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from precision_attention_diffusion_sage_gb300.inputs import make_qkv
    cores = os.cpu_count()
    budget = 150.0 / max(1, args.steps + args.warmup)
    times, flops = [], 0.0
    desc, n = "", 0
    qkv = make_qkv(w)
    for i in range(args.warmup + args.steps):
        f, dt, desc, n = _cpu_oracle_sample(w, budget, qkv)
        if i >= args.warmup:
            times.append(dt)
            flops = f
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "D": w.D,
                       "k_lens": w.k_lens},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--cta-mode", type=int, default=0, choices=[0, 1, 2],
                    help="attention tiles: 0 library choice, 1 one CTA, 2 CTA pairs (cta_group::2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads (a smaller case for profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from dataclasses import replace as _replace
    from precision_attention_diffusion_sage_gb300.inputs import WORKLOADS, make_qkv
    w = WORKLOADS[args.workload]
    if args.heads > 0:
        w = _replace(w, H=args.heads)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from precision_attention_diffusion_sage_gb300 import binding

    def barrier():
        if world > 1:
            dist.barrier()

    q, k, v = make_qkv(w, device="cuda")
    fmt = w.fmt
    B, Nq, H, D = q.shape
    Nk = k.shape[1]
    Nqp, Nkp = binding.pad128(Nq), binding.pad128(Nk)
    k_lens = None if w.k_lens is None else torch.tensor(w.k_lens, dtype=torch.int32, device=dev)
    if fmt == binding.FMT_INT8:
        qq = torch.empty((B, H, Nqp, D), dtype=torch.float16, device=dev)
        qs = torch.empty((B, H, Nqp // 128), dtype=torch.float32, device=dev)
        kq = torch.empty((B, H, Nkp, D), dtype=torch.float16, device=dev)
        ks = torch.empty((B, H, Nkp // 128), dtype=torch.float32, device=dev)
    elif fmt == binding.FMT_FP8:
        qq = torch.empty((B, H, Nqp, D), dtype=torch.uint8, device=dev)
        qs = torch.empty((B, H, Nqp // 128), dtype=torch.float32, device=dev)
        kq = torch.empty((B, H, Nkp, D), dtype=torch.uint8, device=dev)
        ks = torch.empty((B, H, Nkp // 128), dtype=torch.float32, device=dev)
    else:
        qq = torch.empty((B, H, Nqp, D // 2), dtype=torch.uint8, device=dev)
        qs = torch.empty((B, H, Nqp, D // 32), dtype=torch.uint8, device=dev)
        kq = torch.empty((B, H, Nkp, D // 2), dtype=torch.uint8, device=dev)
        ks = torch.empty((B, H, Nkp, D // 32), dtype=torch.uint8, device=dev)
    if fmt == binding.FMT_MXFP4_V4:
        vq = torch.empty((B, H, D, Nkp // 2), dtype=torch.uint8, device=dev)
        vs = torch.empty((B, H, Nkp // 128, D, 4), dtype=torch.uint8, device=dev)
    else:
        vq = torch.empty((B, H, Nkp, D), dtype=torch.uint8, device=dev)
        vs = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    vws = torch.empty(max(16, binding.sage_workspace_bytes(1, fmt, B, H, Nk, Nk)), dtype=torch.uint8,
                      device=dev)
    o = torch.empty((B, Nq, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    aws_n = binding.sage_workspace_bytes(2, fmt, B, H, Nq, Nk, D, args.splits)
    aws = torch.empty(max(16, aws_n), dtype=torch.uint8, device=dev)
    nsplit = binding.attn_splits(B, H, Nq, Nk, args.splits)
    # L2 flush between steps: reading 256 MiB leaves L2 holding clean lines of
    # an unrelated buffer (a write would leave dirty lines whose write-back
    # lands on the next kernel).
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    qm = (torch.empty((B, H, Nqp // 128, D), dtype=torch.float32, device=dev) if w.smooth_q
          else None)
    dsb = (torch.empty((B, H, Nqp // 128, Nkp), dtype=torch.float32, device=dev) if w.smooth_q
           else None)

    def quant_q():
        if w.smooth_q:
            binding.sage_quantize_q_smooth(q, out=qq, scale=qs, q_mean=qm)
        else:
            binding.sage_quantize_qk(q, fmt, out=qq, scale=qs)

    km = torch.empty((B, H, D), dtype=torch.float32, device=dev) if w.smooth_k else None
    kws = (torch.empty(binding.sage_workspace_bytes(3, fmt, B, H, Nk, Nk), dtype=torch.uint8,
                       device=dev) if w.smooth_k else None)

    def quant_k():
        if w.smooth_k:
            binding.sage_quantize_k_smooth(k, lens=k_lens, out=kq, scale=ks, k_mean=km,
                                           workspace=kws)
        else:
            binding.sage_quantize_qk(k, fmt, lens=k_lens, out=kq, scale=ks)

    def quant_v():
        if fmt == binding.FMT_MXFP4_V4:
            binding.sage_quantize_v_mxfp4(v, lens=k_lens, out=vq, scale=vs)
        else:
            binding.sage_quantize_v(v, lens=k_lens, out=vq, scale=vs, workspace=vws)

    def delta_s():
        binding.sage_delta_s(qm, kq, ks, Nq=Nq, Nk=Nk, k_mean=km, out=dsb)

    def attn():
        binding.sage_attn_fwd(fmt, qq, qs, kq, ks, vq, vs, Nq=Nq, Nk=Nk, k_lens=k_lens, out=o,
                              lse=lse, num_splits=args.splits, workspace=aws, k_mean=km,
                              delta_s=dsb, cta_mode=args.cta_mode)

    def quant_qkv():
        binding.sage_quantize_qkv(q, k, v, fmt, k_lens=k_lens, outs=((qq, qs), (kq, ks), (vq, vs)),
                                  workspace=vws)

    # The step: one quantize call for Q, K and V (with smoothing: the three
    # calls it needs, and Q smoothing's dS), then attention. The separate
    # calls are timed as a diagnostic.
    calls = (quant_q, quant_k, quant_v, attn)
    if w.smooth_q:
        quant_step = (quant_q, quant_k, quant_v, delta_s)
    elif w.smooth_k:
        quant_step = (quant_q, quant_k, quant_v)
    else:
        quant_step = (quant_qkv,)
    step_calls = quant_step + (attn,)
    for _ in range(args.warmup):
        for c in calls + step_calls:
            c()
    torch.cuda.synchronize()
    assert binding.sage_last_device_status() == 0

    # The timed step replays two CUDA graphs holding exactly the library's
    # launches (quantize Q, K and V; attention), so the device time carries
    # no host launch gaps. Also timed: each call in a graph of its own (the
    # per-call split; every graph launch adds a few microseconds), and the
    # same calls issued eagerly.
    def capture(fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for fn in fns:
                fn()
        return g

    g_quant, g_attn = capture(quant_step), capture([attn])
    per_call_graphs = [capture([c]) for c in calls]
    for _ in range(args.warmup):
        g_quant.replay()
        g_attn.replay()
        for g in per_call_graphs:
            g.replay()
    torch.cuda.synchronize()
    assert binding.sage_last_device_status() == 0

    def timed(runs):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)]
               for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.sum()
            evs[i][0].record()
            for j, r in enumerate(runs):
                r()
                evs[i][j + 1].record()
        torch.cuda.synchronize()
        barrier()
        # per call: list over steps
        return [[e[j].elapsed_time(e[j + 1]) for e in evs] for j in range(len(runs))]

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    t_quant, t_attn = timed([g_quant.replay, g_attn.replay])
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    assert binding.sage_last_device_status() == 0
    per_call = timed([g.replay for g in per_call_graphs])
    eager_calls = timed(list(step_calls))
    t_quant_eager = [sum(x) for x in zip(*eager_calls[:-1])]
    t_attn_eager = eager_calls[-1]
    assert binding.sage_last_device_status() == 0
    total_ms = sum(t_quant) + sum(t_attn)
    eager_ms = (sum(t_quant_eager) + sum(t_attn_eager)) / args.steps
    total_ms = max_over_ranks(total_ms, world, dev)
    flops = w.flops
    value = replica_throughput(flops, args.steps, total_ms, world)
    attn_ms = statistics.mean(t_attn)
    hbm, p16, peak_kind = _peaks()
    peak = _roofline_peak(p16, fmt)
    achieved = flops / (attn_ms * 1e-3) / 1e12

    # end to end through the public call, host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        host_kw = dict(fmt=fmt, k_lens=w.k_lens, num_splits=args.splits, smooth_k=w.smooth_k,
                       smooth_q=w.smooth_q, cta_mode=args.cta_mode)
        ws_host = torch.empty(binding.sage_attention_host_workspace_bytes(
            w.B, w.Nq, w.Nk, w.H, fmt=fmt, smooth_k=w.smooth_k, smooth_q=w.smooth_q,
            num_splits=args.splits, cta_mode=args.cta_mode, k_lens=w.k_lens is not None),
            dtype=torch.uint8, device=dev)

        def e2e_step():
            # host Q/K/V in, host O/LSE out: head groups are copied in,
            # quantized, attended and copied out by the library, pipelined
            binding.sage_attention_host(qh, kh, vh, out=oh, lse=lh, workspace=ws_host, **host_kw)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        barrier()
        for i in range(args.steps):
            flush.sum()
            ee[i][0].record()
            e2e_step()
            ee[i][1].record()
        torch.cuda.synchronize()
        barrier()
        e_ms = sum(a.elapsed_time(b) for a, b in ee)
        e_ms = max_over_ranks(e_ms, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": replica_throughput(flops, args.steps, e_ms, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = tuple(t.cpu() for t in (q, k, v))
        f, dt, desc, n = _cpu_oracle_sample(w, args.cpu_seconds, host)
        f1, dt1, desc1, _ = _cpu_oracle_sample(w, args.cpu_seconds / 3, host, nthreads=1)
        del host
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": desc, "seconds": dt,
               "value_1core": f1 / dt1 / 1e12, "sample_1core": desc1, "seconds_1core": dt1}

    # Kernels per step: INT8/FP8 fused Q/K/V pass + V encode; MXFP4 formats Q,
    # K, V maxima, V encode; K smoothing Q, four K kernels (maxima, sums,
    # means, encode), V maxima, V encode; then attention (+ split merge).
    if w.smooth_k or w.smooth_q:
        quant_launches = 1 + (4 if w.smooth_k else 1) + 2 + (1 if w.smooth_q else 0)
    elif fmt in (binding.FMT_INT8, binding.FMT_FP8):
        quant_launches = 2
    else:
        quant_launches = 3 if fmt == binding.FMT_MXFP4_V4 else 4
    launches_per_step = quant_launches + 1 + (1 if nsplit > 1 else 0)
    quant_bytes = _quant_bytes(w, Nqp, Nkp)
    # Secondary bound: one exp2 per logit on the MUFU pipe (no FMA-polynomial
    # exponentials are used), at the SM clock sampled during the run.
    nk_sum = sum(w.k_lens) if w.k_lens else w.B * w.Nk
    exp2_count = float(w.H) * w.Nq * nk_sum
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    exp2_ms = exp2_count / (_EX2_PER_CLK_SM * 152 * mhz * 1e6) * 1e3
    nqt = 2 if Nqp >= 256 else 1
    # The library's default (cta_mode 0) is 1-CTA tiles for every shape.
    cta2 = args.cta_mode == 2
    kfmt = 1 if fmt == 3 else fmt   # the rotated MXFP4 format runs the MXFP4 kernel
    # Q smoothing runs the instance that adds dS to the logits (last template flag).
    ds_flag = ",1" if w.smooth_q else ""
    stages = 4 if cta2 else ((2 if nqt == 2 else 3) if kfmt == 0 else 4)
    kernel = f"sage_attn_kernel<{kfmt},{nqt},{stages}{ds_flag}{',0,1' if cta2 else ''}>"
    fmt_names = {0: ("int8+fp8e4m3", "int8_qk_fp8_v"), 1: ("mxfp4+fp8e4m3", "mxfp4_qk_fp8_v"),
                 4: ("mxfp4", "mxfp4_qk_mxfp4_pv"),
                 2: ("fp8e4m3", "fp8_qk_fp8_v"),
                 3: ("mxfp4+fp8e4m3", "hadamard_mxfp4_qk_fp8_v")}
    traffic = _profiled_traffic(kernel, w.name) if args.heads == 0 else None
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": fmt_names[fmt][0], "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "Nq": Nq, "Nk": Nk, "D": D,
                   "k_lens": w.k_lens,
                   "heads_override": args.heads > 0,
                   "format": fmt_names[fmt][1],
                   "k_smoothing": w.smooth_k,
                   "q_smoothing": w.smooth_q,
                   "splits": nsplit,
                   "l2": "flushed between steps (256 MiB read outside the timed events)",
                   "launch": ("two CUDA graphs per step: the quantize call (sage_quantize_qkv; with K "
                              "smoothing the three quantize calls) and the attention call"),
                   "cta": (("2-CTA tiles (cta_group::2, clusters of two CTAs, M = 256 rows), "
                            if cta2 else "1-CTA tiles (cta_group::1), ")
                           + f"{nqt} query tile(s) of 128 rows per CTA, one MMA warp per tile"),
                   "parallelism": f"replicas x{world}"},
        "eager_ms_per_step": eager_ms,
        "attn_only_tflops": achieved,
        "quant_ms_per_step": statistics.mean(t_quant),
        "quant_separate_calls_ms": [round(statistics.mean(c), 5) for c in per_call[:3]],
        "attn_ms_per_step": attn_ms,
        "quant_gbs": quant_bytes / (statistics.mean(t_quant) * 1e-3) / 1e9,
        "quant_hbm_frac": quant_bytes / (statistics.mean(t_quant) * 1e-3) / 1e9 / hbm,
        "exp2_bound": {"exp2_per_step": exp2_count, "mufu_ex2_per_clk_sm": _EX2_PER_CLK_SM,
                       "ms": exp2_ms, "vs_tensor_bound_ms": flops / (peak * 1e12) * 1e3},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": None if traffic is None else traffic,
                     "algorithmic_flops_per_launch": flops,
                     "peak_basis": (f"{peak_kind} bf16 {p16} TFLOP/s x nominal ratios: Q K^T "
                                    f"{ {0: 'fp16 x1', 1: 'fp4 x6', 2: 'fp8 x2', 3: 'fp4 x6', 4: 'fp4 x6'}[fmt] }, "
                                    f"P V { 'fp4 x6' if fmt == 4 else 'fp8 x2' }, "
                                    f"harmonic combination"),
                     "kernel": kernel,
                     "peak_at_sampled_clock": _clock_peak(fmt, mhz),
                     "frac_at_sampled_clock": achieved / _clock_peak(fmt, mhz),
                     "sampled_clock_basis": (f"measured tcgen05 FLOP/clk/SM (f16 8192, f8 16384, "
                                             f"f4 32768) x {_SMS} SMs x median SM clock {mhz} MHz "
                                             f"sampled during the timed region; informational")},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk, "wall_s": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
