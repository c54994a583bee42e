"""Benchmark: fwd and fwd+bwd TFLOPS of exact attention at D=512, N=8192, bf16.

One step = the whole hot path on one batch of synthetic input already
resident in HBM: forward (O, LSE) then backward (preprocess, dK/dV, dQ), all
through the C ABI. FLOPs follow the usual convention: forward
4*B*Hq*Nq*Nkv*D, backward 2.5x that, both halved when causal.

Prints ONE JSON line (rank 0). Multi-GPU runs (torchrun) give every rank the
same per-GPU workload (weak scaling; no data-path collective) and report the
slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config headline|tiny|gqa|sweep320|sweep640|sweep1024|varlen|decode|fp8]

--config decode times the split-KV decode forward instead (GB/s of the
bytes it must move; a step of it takes well under a millisecond, so give it
a few thousand --steps for the clock samples to fall inside the timed region).
--config fp8 times the e4m3 forward (ffpa_fwd_fp8: quantization + attention).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd & fwd+bwd TFLOPS, D=512 N=8192 bf16 (1×GB300), % of BF16 tensor peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: a timed region of >= 2 s for the chosen workload)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="headline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other workloads measured beside the headline in the default run")
    ap.add_argument("--all", action="store_true",
                    help="one line per workload, decode and fp8 included (parity-size cases excluded)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override Hq=Hkv (profiling a smaller case of the same kernels)")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override Nq=Nkv of a dense workload (the same recipe at another sequence length)")
    return ap.parse_args()


def workload(name):
    from head_dim_flash_gb300 import workloads as W

    table = {"headline": W.HEADLINE, "tiny": W.TINY, "gqa": W.GQA_CAUSAL,
             "sweep320": W.SWEEP[0], "sweep640": W.SWEEP[1], "sweep1024": W.SWEEP[2], "varlen": W.VARLEN,
             "decode": W.DECODE, "fp8": W.FP8}
    if name not in table:
        raise SystemExit(f"unknown config {name}; choose from {sorted(table)}")
    return table[name]


def flops(w):
    if w.varlen:
        f = sum(4.0 * w.Hq * n * n * w.D for n in w.seqlens)
    else:
        f = 4.0 * w.B * w.Hq * w.Nq * w.Nkv * w.D
    if w.causal:
        f *= 0.5
    return f, 2.5 * f


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
    return rank, world, local


def slowest_rank_ms(ms: float, world: int, device="cpu") -> float:
    """Max over ranks of a timed region (ms): the whole job is as fast as its slowest rank."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(per_rank_flops: float, world: int, ms: float) -> float:
    """Weak scaling: every rank runs the same per-GPU work; value = all ranks' FLOPs / slowest time."""
    return world * per_rank_flops / (ms / 1e3) / 1e12


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


def cpu_baseline(w, inp, n_rows=8192):
    """Times the fp64 oracle on a bounded sample of the workload: forward and
    backward of `n_rows` query rows of head 0 of batch 0 against all its keys
    (`inp` are the workload's inputs, made once by the caller).
    Returns (tflops, seconds, cores, description)."""
    import oracle

    if w.varlen:
        # packed [T, H, D]: the first sequence, head 0, as a [1, 1, N, D] problem
        n_keys = w.seqlens[0]
        rows = min(n_rows, n_keys)

        def dense(x, n):
            return x[:n, 0:1, :].permute(1, 0, 2).unsqueeze(0).contiguous()

        q, do = dense(inp["q"], rows), dense(inp["dO"], rows)
        k, v = dense(inp["k"], n_keys), dense(inp["v"], n_keys)
    else:
        n_keys = w.Nkv
        rows = min(n_rows, w.Nq)
        q = inp["q"][0:1, 0:1, :rows]
        k = inp["k"][0:1, 0:1]
        v = inp["v"][0:1, 0:1]
        do = inp["dO"][0:1, 0:1, :rows]
    oracle.build()
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, False, w.scale)
    oracle.attention_bwd(q, k, v, do, False, w.scale)
    dt = time.perf_counter() - t0
    f = 3.5 * 4.0 * rows * n_keys * w.D  # fwd + bwd counted flops of the sample
    desc = (f"fwd+bwd of {rows} query rows x {n_keys} keys of head 0 (D={w.D}, non-causal sample"
            f"{', first sequence' if w.varlen else ''}), fp64 C oracle, OpenMP")
    return f / dt / 1e12, dt, cores, desc


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an
# ncu capture, keyed by (workload, kernel), with the hash of the sources the
# capture ran; the figure is reported only while those sources still hash
# the same (the ncu summaries under profiles/ give the commands and the raw
# counters).
PAIR_SOURCES = ("xchg.cu", "xchg2.cu", "ptx.cuh", "tile_common.cuh", "kernels.h", "bwd.cu")
DECODE_SOURCES = ("decode.cu", "ptx.cuh", "tile_common.cuh", "kernels.h")
FP8_SOURCES = ("xchg2.cu", "fp8.cu", "ptx.cuh", "tile_common.cuh", "kernels.h", "host.cu")
TRAFFIC = {
    # dK (also storing P^T and dS^T) at 16 heads (753,212,672 + 4,365,639,168 bytes) scaled to 32
    ("dense B1 H32 N8192 D512 bf16", "dk"): {"bytes": 10237703680, "files": PAIR_SOURCES,
                                             "sources": "4688995f040b0615"},
    # one ffpa_decode_fwd call: split kernel + combine (means over six calls)
    ("decode B8 Hq32 Hkv8 Nq1 Nkv16384 D512 bf16", "decode"): {"bytes": 2156570368, "files": DECODE_SOURCES,
                                                                "sources": "6e118bc1610051ae"},
    # the e4m3 attention kernel (reads q8, k8, V^T codes; writes O, LSE)
    ("fp8 forward dense B1 H32 N8192 D512 (bf16 in, e4m3 compute)", "fp8"): {"bytes": 641944474,
                                                                             "files": FP8_SOURCES,
                                                                             "sources": "1f4f6f4eb7b809e7"},
}


def kernel_source_hash(files=PAIR_SOURCES):
    import hashlib

    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "head_dim_flash_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(w, kernel):
    rec = TRAFFIC.get((w.name, kernel))
    if rec is None or rec["sources"] != kernel_source_hash(rec["files"]):
        return None
    return rec["bytes"]


def run_reference(args):
    """The oracle timed as the reference arm (bounded sample per step)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args.config)
    import oracle
    from head_dim_flash_gb300 import workloads as W

    oracle.build()
    inp = W.make_inputs(w)
    rows = 256
    times = []
    for i in range(args.warmup + args.steps):
        tf, dt, cores, desc = cpu_baseline(w, inp, n_rows=rows)
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    f = 3.5 * 4.0 * rows * w.Nkv * w.D
    value = f / (ms / 1e3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": f"{rows} query rows of head 0"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_METRIC = "decode forward (split-KV): algorithmic HBM GB/s (q, K/V cache, O, LSE), D=512 bf16 (1×GB300)"


def decode_bytes(w):
    """Bytes the decode forward must move: read q, K, V; write O (16-bit) and LSE (fp32)."""
    q = w.B * w.Hq * w.Nq * w.D * 2
    kv = 2 * w.B * w.Hkv * w.Nkv * w.D * 2
    return q + kv + q + w.B * w.Hq * w.Nq * 4


def run_decode(args, w):
    """Decode workload: one ffpa_decode_fwd call per step (split kernel + combine)."""
    import torch

    from head_dim_flash_gb300 import api
    from head_dim_flash_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = W.make_inputs(w, with_grad_out=False)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    from head_dim_flash_gb300 import _ffi

    ws_bytes = _ffi.ffpa_decode_workspace_bytes(api._dt(q), w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.decode_fwd(q, k, v, w.causal, w.scale, out=o, lse=lse, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    api.get_status()
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for ev in events:
            ev[0].record(stream)
            step()
            ev[1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    api.get_status()
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in events)
    ms_step = slowest_rank_ms(start.elapsed_time(end), world, dev) / args.steps
    nbytes = decode_bytes(w)
    value = world * nbytes / (ms_step / 1e3) / 1e9
    pk = peaks()
    achieved = nbytes / (call_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": "decode (split kernel + combine, one ffpa_decode_fwd call)",
            "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
            "traffic": measured_traffic(w, "decode"), "peak_source": f"{pk['source']} copy bandwidth"}
    e2e = None
    if not args.no_e2e:
        # the K/V cache stays resident (as in serving); each step copies the
        # new query rows host->device and reads O and LSE back
        qh = inp["q"].pin_memory()
        oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        qd = torch.empty_like(q)

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            api.decode_fwd(qd, k, v, w.causal, w.scale, out=o, lse=lse, workspace=ws)
            oh.copy_(o, non_blocking=True)
            lh.copy_(lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        n = max(1, args.steps)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        ems = s0.elapsed_time(s1) / n
        e2e = {"value": world * nbytes / (ems / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
               "h2d_bytes_per_step": qh.numel() * qh.element_size(),
               "d2h_bytes_per_step": oh.numel() * oh.element_size() + lh.numel() * lh.element_size(),
               "note": "K/V cache resident on the device"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = decode_cpu_baseline(w, inp)
    if rank == 0:
        line = {
            "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D,
                       "causal": w.causal, "l2": "K/V cache larger than L2 (2.1 GB)"},
            "rows_per_s": world * w.B * w.Hq * w.Nq / (ms_step / 1e3),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
            "gpu_launches": 2 * args.steps,  # split kernel + combine per step
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def decode_cpu_baseline(w, inp):
    """The fp64 oracle on the whole decode workload, one batch entry at a time."""
    import oracle

    oracle.build()
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    for b in range(w.B):
        oracle.attention_fwd(inp["q"][b:b + 1], inp["k"][b:b + 1], inp["v"][b:b + 1], w.causal, w.scale)
    dt = time.perf_counter() - t0
    return {"value": decode_bytes(w) / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle", "seconds": dt,
            "sample": f"the whole workload ({w.B} x {w.Hq} heads x {w.Nq} rows x {w.Nkv} keys, D={w.D}), "
                      "fp64 C oracle, one batch entry per call"}


FP8_METRIC = "fp8 (e4m3) forward TFLOPS, D=512 N=8192, bf16 in/out (1×GB300), % of the fp8 tensor peak"


def run_fp8(args, w):
    """FP8 workload: one ffpa_fwd_fp8 call per step (quantization pass + attention)."""
    import torch

    from head_dim_flash_gb300 import api
    from head_dim_flash_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = W.make_inputs(w, with_grad_out=False)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    ws = api.fp8_workspace(q, k)
    stream = torch.cuda.current_stream(dev)
    f_fwd = flops(w)[0]

    def step():
        api.fwd_fp8(q, k, v, w.causal, w.scale, out=o, lse=lse, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    api.get_status()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    api.get_status()
    ms_step = slowest_rank_ms(start.elapsed_time(end), world, dev) / args.steps
    value = job_throughput(f_fwd, world, ms_step)

    # per-kernel pass: the quantization alone, the attention alone (from the workspace)
    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a_, b_ in evs:
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)

    n_k = min(args.steps, 10)
    quant_ms = timed(lambda: api.fp8_quantize(q, k, v, workspace=ws), n_k)
    attn_ms = timed(lambda: api.fwd_fp8_quantized(ws, q.shape, k.shape, q.dtype, w.causal, w.scale, out=o, lse=lse),
                    n_k)
    api.get_status()
    pk = peaks()
    # the attention kernel is timed launched alone (a burst): the burst bf16 peak x 2
    peak8 = 2.0 * pk["bf16_tflops"]
    achieved = f_fwd / (attn_ms / 1e3) / 1e12
    clocks = clk.summary()
    at8 = at_clock(achieved / 2.0, clocks.get("sm_mhz"))  # e4m3 runs at twice the 16-bit rate per clock
    roof = {"bound": "tensor", "kernel": "fp8 pair forward (attention, from the quantized workspace)",
            "achieved": achieved, "peak": peak8, "unit": "TFLOP/s", "frac": achieved / peak8,
            "traffic": measured_traffic(w, "fp8"),
            "peak_source": f"{pk['source']} burst bf16 x 2 (nominal e4m3 / bf16 dense ratio 4.5 / 2.25)",
            "at_clock": None if at8 is None else {"sm_mhz": at8["sm_mhz"], "peak_tflops": 2 * at8["peak_tflops"],
                                                  "frac": at8["frac"]}}
    qbytes = 3 * w.B * w.Hq * w.Nq * w.D * 2 * 2 + 3 * w.B * w.Hq * w.Nq * w.D  # read twice, write codes

    e2e = None
    if not args.no_e2e:
        # q, k, v in and O, LSE out every step; the quantization workspace is
        # reused (the steps run in order on the compute stream)
        host = {n: inp[n].pin_memory() for n in ("q", "k", "v")}

        def call(x):
            o_, l_ = api.fwd_fp8(x["q"], x["k"], x["v"], w.causal, w.scale, workspace=ws)
            return {"o": o_, "lse": l_}

        ems, h2d, d2h = overlapped_e2e(dev, stream, host, call, max(1, min(args.steps, 30)))
        e2e = {"value": world * f_fwd / (ems / 1e3) / 1e12, "unit": "TFLOPS", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "overlap": E2E_OVERLAP}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = fp8_cpu_baseline(w, inp)
    if rank == 0:
        line = {
            "metric": FP8_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate; bf16 in/out)", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D,
                       "causal": w.causal, "l2": "inputs larger than L2 (each of q/k/v 268 MB)"},
            "kernel_ms": {"quantize": quant_ms, "attention": attn_ms},
            "quantize_gbs": qbytes / (quant_ms / 1e3) / 1e9,
            "pct_peak_fp8": 100 * value / world / peak8,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 4 * args.steps,  # amax, q/k codes, V^T codes, attention per step
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def fp8_cpu_baseline(w, inp, n_rows=1024):
    """The oracle's FP8 reference on a bounded sample: quantization of head 0
    and the attention of `n_rows` of its query rows against all keys."""
    import oracle
    from oracle import fp8 as ofp8

    oracle.build()
    cores = oracle.num_threads()
    rows = list(range(min(n_rows, w.Nq)))
    t0 = time.perf_counter()
    qd = ofp8.dequantize(*ofp8.quantize(inp["q"][0:1, 0:1]))
    kd = ofp8.dequantize(*ofp8.quantize(inp["k"][0:1, 0:1]))
    vd = ofp8.dequantize(*ofp8.quantize(inp["v"][0:1, 0:1]))
    oracle.attention_fwd_rows(qd[0, 0], kd[0, 0], vd[0, 0], rows, w.causal, w.scale)
    dt = time.perf_counter() - t0
    f = 4.0 * len(rows) * w.Nkv * w.D
    return {"value": f / dt / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "seconds": dt,
            "sample": f"e4m3 quantization of head 0 and the fp64 attention of {len(rows)} of its query rows x "
                      f"{w.Nkv} keys (D={w.D})"}


def build_steps(w, dev, stream, inp):
    """The workload's step on device-resident inputs: one forward call and one
    backward call (the user's path; the backward's kernels overlap their
    neighbours' tails). Returns a dict with `step(ev)` (records ev[0..2]
    around fwd / bwd when given), `kernel_step(ev)` and `kernel_names` for the
    per-kernel pass (dense only), and `ds_path` (stored-tile backward)."""
    import torch

    from head_dim_flash_gb300 import _ffi, api

    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "dO"))
    o = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    out = {"kernel_step": None, "kernel_names": None}
    if w.varlen:
        # packed batch: forward and the whole backward through the varlen entry points
        cu = inp["cu_seqlens"].to(dev)
        mx = max(w.seqlens)
        # the path varlen_bwd's own workspace (within the default budget) takes
        sizes = (_ffi.BF16 if w.dtype == torch.bfloat16 else _ffi.FP16, len(w.seqlens), sum(w.seqlens),
                 sum(w.seqlens), mx, mx, w.Hq, w.Hkv, w.D)
        n_ws = api.varlen_workspace_bytes(q, k, cu, mx, mx, w.causal)
        out.update(workspace_path(n_ws, int(_ffi.ffpa_varlen_bwd_workspace_bytes(*sizes)),
                                  int(_ffi.ffpa_varlen_bwd_workspace_bytes_ds(*sizes, int(w.causal)))))
        state = {}

        def step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            state["o"], state["lse"] = api.varlen_fwd(q, k, v, cu, cu, mx, mx, w.causal, w.scale)
            if ev is not None:
                ev[1].record(stream)
            api.varlen_bwd(q, k, v, state["o"], state["lse"], do, cu, cu, mx, mx, w.causal, w.scale)
            if ev is not None:
                ev[2].record(stream)
    else:
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        # the default workspace (within api.BWD_WORKSPACE_BUDGET): with every head's
        # tiles, dK also stores P^T and dS^T and dV and dQ are one GEMM each over
        # them; with a chunk of kv groups' tiles the same runs chunk by chunk
        ws = api.bwd_workspace(q, k, w.causal)
        small = api.bwd_workspace_bytes(q, k)
        out.update(workspace_path(ws.numel(), small, api.bwd_workspace_bytes(q, k, w.causal)))
        ds_path = out["ds_path"]
        if out["chunked"]:
            # kv groups per chunk: the largest evened-out count whose two tile sets fit
            group = w.B * (w.Hq // w.Hkv) * w.Nkv * ((w.Nq + 7) // 8 * 8) * 2
            ng = max(g for g in range(1, w.Hkv + 1) if small + (g * group + 255) // 256 * 256 + g * group <= ws.numel())
            chunks = -(-w.Hkv // ng)
            out["chunks"] = chunks
            out["bwd_path"] += f": {chunks} chunks of {-(-w.Hkv // chunks)} kv groups"

        def step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            api.fwd(q, k, v, w.causal, w.scale, out=o, lse=lse)
            if ev is not None:
                ev[1].record(stream)
            api.bwd(q, k, v, o, lse, do, w.causal, w.scale, workspace=ws, dq=dq, dk=dk, dv=dv)
            if ev is not None:
                ev[2].record(stream)

        # per-kernel durations (a second timed pass, one launch per call:
        # preprocess | dV | dK | dQ are ffpa_bwd_stages bits 0, 1, 3, then 2, or 4
        # for the dQ GEMM over the dS that the dK launch just stored; with bit 5
        # dK also stores P and runs first, and dV is the GEMM over that P, as in
        # the full call)
        kernel_names = ("fwd", "preprocess", "dk", "dv", "dq") if ds_path else ("fwd", "preprocess", "dv", "dk", "dq")
        stage_bits = (1, 8 | 32, 2 | 32, 16) if ds_path else (1, 2, 8, 4)

        def kernel_step(ev):
            ev[0].record(stream)
            api.fwd(q, k, v, w.causal, w.scale, out=o, lse=lse)
            for i, bit in enumerate(stage_bits):
                ev[i + 1].record(stream)
                api.bwd(q, k, v, o, lse, do, w.causal, w.scale, workspace=ws, dq=dq, dk=dk, dv=dv, stages=bit)
            ev[5].record(stream)

        if not out["chunked"]:  # the stage bits time the one-chunk layout only
            out["kernel_step"], out["kernel_names"] = kernel_step, kernel_names
    out["step"] = step
    return out


def workspace_path(n_ws, small, full):
    """Which backward a workspace of n_ws bytes runs (small: row statistics
    only; full: every head's stored tiles)."""
    if full > small and n_ws >= full:
        path, chunked = "stored tiles, every head at once", False
    elif full > small and n_ws > small:
        path, chunked = "stored tiles in chunks of kv groups (workspace below the every-head size)", True
    else:
        path, chunked = "recompute (no stored tiles)", False
    return {"ds_path": n_ws > small and full > small, "chunked": chunked, "bwd_path": path,
            "workspace_bytes": int(n_ws)}


def time_steps(st, steps, warmup, stream, world, local, dev):
    """Warm-up, then exactly `steps` timed steps between barriers and device
    syncs (CUDA events on the launch stream), with the SM clocks sampled
    meanwhile. Returns (ms per step (max over ranks), mean fwd / bwd ms, clocks)."""
    import torch

    from head_dim_flash_gb300 import api

    for _ in range(warmup):
        st["step"]()
    torch.cuda.synchronize()
    api.get_status()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            st["step"](events[i])
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    api.get_status()
    fwd_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in events)
    bwd_ms = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in events)
    ms_step = slowest_rank_ms(start.elapsed_time(end), world, dev) / steps
    return ms_step, fwd_ms, bwd_ms, clk.summary()


def kernel_times(st, stream, n=10):
    """Per-kernel CUDA-event times, each kernel launched alone (dense workloads)."""
    import torch

    from head_dim_flash_gb300 import api

    names = st["kernel_names"]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n)]
    st["kernel_step"](kev[0])
    torch.cuda.synchronize()
    for ev in kev:
        st["kernel_step"](ev)
    torch.cuda.synchronize()
    api.get_status()
    return {nm: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in kev) for i, nm in enumerate(names)}


def num_sms():
    import torch

    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


# dense bf16 / fp16 tensor FLOPs per SM per clock of a 5th-generation tensor
# core SM (4 x 2048): the clock-for-clock denominator
TENSOR_FLOPS_PER_SM_CLK = 8192


def at_clock(tflops, sm_mhz):
    """Achieved TFLOP/s against the tensor rate at the sampled median SM clock."""
    if not sm_mhz:
        return None
    peak = num_sms() * TENSOR_FLOPS_PER_SM_CLK * sm_mhz * 1e6 / 1e12
    return {"sm_mhz": sm_mhz, "peak_tflops": peak, "frac": tflops / peak,
            "note": f"{num_sms()} SMs x {TENSOR_FLOPS_PER_SM_CLK} dense 16-bit FLOP/clk x median sampled SM clock"}


# default timed steps per workload: a timed region of >= 2 s, so that the
# clock sampler sees the steady power state
DEFAULT_STEPS = {"headline": 200, "tiny": 2000, "gqa": 200, "sweep320": 1000, "sweep640": 600, "sweep1024": 400,
                 "varlen": 250, "decode": 6000, "fp8": 600}
# the workloads measured beside the headline in the default run (one GPU):
# the other configs of the metric, each with a short timed region
OTHER_WORKLOADS = ("gqa", "sweep320", "sweep640", "sweep1024", "varlen")


def measure_other(name, dev, stream, pk, steps=30):
    """fwd / bwd / fwd+bwd TFLOPS of another workload in this run (the same
    step and timing rules as the headline, a shorter timed region)."""
    import gc

    import torch

    from head_dim_flash_gb300 import workloads as W

    w = workload(name)
    f_fwd, f_bwd = flops(w)
    st = build_steps(w, dev, stream, W.make_inputs(w))
    ms_step, fwd_ms, bwd_ms, clocks = time_steps(st, steps, 3, stream, 1, dev.index or 0, dev)
    rec = {"workload": w.name, "steps": steps, "ms_per_step": ms_step,
           "tflops": (f_fwd + f_bwd) / (ms_step / 1e3) / 1e12,
           "fwd": {"ms": fwd_ms, "tflops": f_fwd / (fwd_ms / 1e3) / 1e12},
           "bwd": {"ms": bwd_ms, "tflops": f_bwd / (bwd_ms / 1e3) / 1e12},
           "bwd_path": st["bwd_path"], "bwd_workspace_bytes": st["workspace_bytes"], "clocks": clocks}
    rec["pct_peak_burst"] = 100 * rec["tflops"] / pk["bf16_tflops"]
    if w.causal and not w.varlen and w.Nq != w.Nkv:
        legal = legal_fraction(w.Nq, w.Nkv)
        rec["executed_fraction_of_dense"] = legal
        rec["note"] = (f"FLOPs counted halved for causal; the legal pairs are {legal:.4f} of dense, so the "
                       f"legal-pair rate is {rec['tflops'] * legal / 0.5:.0f} TFLOPS")
    del st
    gc.collect()
    torch.cuda.empty_cache()
    return rec


def legal_fraction(nq, nkv):
    """Share of the nq x nkv score matrix that the bottom-right causal mask keeps."""
    off = nkv - nq
    legal = sum(max(0, min(nkv, i + off + 1)) for i in range(nq))
    return legal / (nq * nkv)


def run_ours(args):
    import torch

    from head_dim_flash_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.config)
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.config, 200)
    if args.config == "decode":
        return run_decode(args, w)
    if args.config == "fp8":
        return run_fp8(args, w)
    if args.heads:
        import dataclasses

        g = w.Hq // w.Hkv
        w = dataclasses.replace(w, name=w.name.replace(f"H{w.Hq}", f"H{args.heads}") + f" (heads={args.heads})",
                                Hq=args.heads, Hkv=max(1, args.heads // g))
    if args.seqlen and not w.varlen:
        import dataclasses

        w = dataclasses.replace(w, name=w.name.replace(f"N{w.Nq}", f"N{args.seqlen}"), Nq=args.seqlen,
                                Nkv=args.seqlen)
    f_fwd, f_bwd = flops(w)
    inp = W.make_inputs(w)
    stream = torch.cuda.current_stream(dev)
    st = build_steps(w, dev, stream, inp)
    ds_path = st["ds_path"]
    bwd_path = {"bwd_path": st["bwd_path"], "bwd_workspace_bytes": st["workspace_bytes"]}
    st_chunks = st.get("chunks", 1)
    warmup = max(args.warmup, 3)
    ms_step, fwd_ms, bwd_ms, clocks = time_steps(st, args.steps, warmup, stream, world, local, dev)
    per_ms = {"fwd": fwd_ms, "bwd": bwd_ms}
    if st["kernel_step"] is not None:
        per_ms = kernel_times(st, stream, n=min(args.steps, 10))
    value = job_throughput(f_fwd + f_bwd, world, ms_step)
    pk = peaks()

    # roofline of the dominant kernel (largest time share); algorithmic flops
    # per launch = the GEMMs it runs: fwd 2 (S, PV), dV 2 (S, dV) or 1 on the
    # stored P, dK 3 (S, dP, dK), dQ 3 (S, dP, dQ) or 1 on the stored dS, each
    # 2*B*Hq*Nq*Nkv*D (halved causal)
    gemm = f_fwd / 2.0
    if st["kernel_step"] is None:
        # bwd: preprocess + dK (3) + dV (1) + dQ (1) units on the stored tiles, else
        # preprocess + dV (2) + dK (3) + dQ (3)
        algo = {"fwd": 2 * gemm, "bwd": (5 if ds_path else 8) * gemm}
    else:
        algo = {"fwd": 2 * gemm, "dv": (1 if ds_path else 2) * gemm, "dk": 3 * gemm,
                "dq": (1 if ds_path else 3) * gemm}
    dom = max(algo, key=lambda n: per_ms[n])
    achieved = algo[dom] / (per_ms[dom] / 1e3) / 1e12
    # a kernel launched alone (the per-kernel pass) is a burst: the burst peak
    # applies; a fwd / bwd breakdown comes from the timed region itself
    alone = st["kernel_step"] is not None  # the per-kernel pass ran
    peak = pk["bf16_tflops"] if alone else pk["bf16_tflops_sustained"]
    roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": measured_traffic(w, dom),
            "peak_source": (f"{pk['source']} burst bf16 (the kernel is timed launched alone)" if alone
                            else f"{pk['source']} sustained bf16 (timed inside the steps)"),
            "at_clock": at_clock(achieved, clocks.get("sm_mhz"))}
    if dom == "dk" and alone:
        # bytes the dK launch must move (Q, dO, K, V read; dK written), and the
        # stored-tile writes it adds (the stored-tile backward's trade of memory
        # for FLOPs, not work of the method)
        e = 2
        roof["algorithmic_bytes"] = e * w.D * (2 * w.B * w.Hq * w.Nq + 3 * w.B * w.Hkv * w.Nkv)
        roof["stored_tile_bytes"] = 2 * e * w.B * w.Hq * w.Nkv * ((w.Nq + 7) // 8 * 8) if ds_path else 0
    kernels = {}
    for n, ms in per_ms.items():
        if n in algo:
            tf = algo[n] / (ms / 1e3) / 1e12
            kernels[n] = {"ms": ms, "tflops": tf, "frac_burst": tf / pk["bf16_tflops"],
                          "at_clock": at_clock(tf, clocks.get("sm_mhz"))}

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(w, args, dev, stream, inp, f_fwd + f_bwd, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, cores, desc = cpu_baseline(w, inp)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc, "seconds": dt}

    others = None
    if world == 1 and not args.no_others and args.config == "headline" and not args.heads and not args.seqlen:
        del st, inp
        import gc

        gc.collect()
        torch.cuda.empty_cache()
        others = {n: measure_other(n, dev, stream, pk) for n in OTHER_WORKLOADS}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype.__repr__().endswith("bfloat16") else "fp16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D,
                       "causal": w.causal, "l2": "inputs larger than L2 (each of q/k/v/dO > 129 MB)"
                       if w.B * w.Hq * w.Nq * w.D * 2 > 129e6 else "inputs smaller than L2 (parity-size case)"},
            "fwd": {"tflops": world * f_fwd / (fwd_ms / 1e3) / 1e12, "ms": fwd_ms,
                    "pct_peak_burst": 100 * f_fwd / (fwd_ms / 1e3) / 1e12 / pk["bf16_tflops"],
                    "at_clock": at_clock(f_fwd / (fwd_ms / 1e3) / 1e12, clocks.get("sm_mhz"))},
            "bwd": {"tflops": world * f_bwd / (bwd_ms / 1e3) / 1e12, "ms": bwd_ms,
                    "pct_peak_burst": 100 * f_bwd / (bwd_ms / 1e3) / 1e12 / pk["bf16_tflops"],
                    "at_clock": at_clock(f_bwd / (bwd_ms / 1e3) / 1e12, clocks.get("sm_mhz"))},
            "kernel_ms": per_ms, "kernels": kernels,
            "dq_path": ("one GEMM over the dS stored by the dK launch" if ds_path
                        else "S and dP recomputed"),
            "dv_path": ("one GEMM over the P^T stored by the dK launch" if ds_path
                        else "S^T recomputed"),
            **bwd_path,
            "kernel_ms_note": "each kernel launched alone (one call per stage), after the timed region"
            if alone else "fwd and bwd calls of the timed region",
            "pct_peak_burst": 100 * value / world / pk["bf16_tflops"],
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            # fwd, preprocess, then dK, dV, dQ once, or per chunk of kv groups
            "gpu_launches": (2 + 3 * st_chunks) * args.steps,
            "other_workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def overlapped_e2e(dev, stream, host, call, n):
    """Steps through the public API from pinned host buffers, as a training or
    serving loop runs them: each step copies its inputs (`host`) to the
    device, runs `call` on them (which returns the step's outputs by name) and
    reads every output back. The copies run on two copy streams, into two
    device input buffers, so that step i+1's inputs move in and step i's
    outputs move out while the GPU computes (the C2C link is full duplex).
    The timed region starts before the first input copy and ends after the
    last output copy. Returns (ms per step, h2d bytes, d2h bytes per step)."""
    import torch

    bufs = [{k: torch.empty_like(t, device=dev) for k, t in host.items()} for _ in range(2)]
    out_h = {}  # pinned host copies of the outputs, allocated at the first step
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]  # inputs of buffer b landed
    buf_free = [None, None]                            # last step that read buffer b is done

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if buf_free[b] is not None:
                s_in.wait_event(buf_free[b])
            for k in host:
                bufs[b][k].copy_(host[k], non_blocking=True)
            in_ready[b].record(s_in)

    def compute(i):
        b = i % 2
        stream.wait_event(in_ready[b])
        outs = call(bufs[b])
        done = torch.cuda.Event()
        done.record(stream)
        buf_free[b] = done
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            for k, g in outs.items():
                if k not in out_h:
                    out_h[k] = torch.empty(g.shape, dtype=g.dtype).pin_memory()
                g.record_stream(s_out)  # not reused before the copy has read it
                out_h[k].copy_(g, non_blocking=True)

    def run(m, start=None):
        if start is not None:
            s_in.wait_event(start)
            s_out.wait_event(start)
        copy_in(0)
        for i in range(m):
            if i + 1 < m:
                copy_in(i + 1)
            compute(i)
        stream.wait_stream(s_out)

    run(2)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    run(n, start=s)
    e.record(stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_h.values())
    return s.elapsed_time(e) / n, h2d, d2h


E2E_OVERLAP = ("double-buffered inputs; copies on two side streams overlap the compute of the "
               "neighbouring steps; first copy-in and last copy-out inside the timed region")


def measure_e2e(w, args, dev, stream, inp, step_flops, world):
    """Same metric through the public API with pinned host buffers: every step
    copies q, k, v, dO host->device and reads dq, dk, dv back (overlapped_e2e)."""
    from head_dim_flash_gb300 import api

    names = ("q", "k", "v", "dO") + (("cu_seqlens",) if w.varlen else ())
    host = {n: inp[n].pin_memory() for n in names}

    def call(x):
        if w.varlen:
            cu, mx = x["cu_seqlens"], max(w.seqlens)
            o, lse = api.varlen_fwd(x["q"], x["k"], x["v"], cu, cu, mx, mx, w.causal, w.scale)
            grads = api.varlen_bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], cu, cu, mx, mx, w.causal, w.scale)
        else:
            o, lse = api.fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
            grads = api.bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], w.causal, w.scale)
        return dict(zip(("dq", "dk", "dv"), grads))

    # 30 steps: the first copy-in and the last copy-out (a few ms) that no
    # compute overlaps are spread over a run of training-loop length
    ms, h2d, d2h = overlapped_e2e(dev, stream, host, call, max(1, min(args.steps, 30)))
    return {"value": world * step_flops / (ms / 1e3) / 1e12, "unit": "TFLOPS", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "overlap": E2E_OVERLAP}


def main():
    args = parse()
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 5
        run_reference(args)
        return
    from head_dim_flash_gb300 import build

    build.build()
    if args.all:
        steps = args.steps
        for name in ("headline", "gqa", "sweep320", "sweep640", "sweep1024", "varlen", "decode", "fp8"):
            args.config, args.steps, args.no_others = name, steps, True
            run_ours(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
