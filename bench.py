#!/usr/bin/env python3
"""GDN / KDA mixer forward + backward throughput on GB300, and its roofline.

One step = one forward and one backward pass of the mixer over one batch of
synthetic inputs (every step of the chunkwise method: gate prep, decayed
K K^T, the triangular solve, WY factors, outputs, the inter-chunk state
recurrence, the reverse chunk scan and the gate gradients).  The forward
keeps each chunk's entry state and solve result in a saved context that the
backward reads (gdn_fwd_save / gdn_bwd_saved); the step with the backward
recomputing them is timed beside it and reported as "recompute_variant".

Default workload: GDN, B=16, T=2048, H=8, dk=dv=128, chunk 64, bf16 inputs
with fp32 state (the 300M-model pre-training shape).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  (default K: 1000 GDN steps, about 0.6 s timed, so that the clock samples
  fall inside the timed region; 5 KDA steps; 5000 decode steps; 20 for the
  reference arm)
  python bench.py --workload gdn_decode   # single-token decode step
  python bench.py --workload gdn_1m       # 1M-token forward
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

With N > 1 (launched by torch.distributed.run) every rank runs its own batch
(independent sequences, no exchange: weak scaling) and rank 0 reports the
aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_bwd_gb300 import workloads as W  # noqa: E402

METRIC = "GDN/KDA mixer fwd+bwd tokens/s on 1 GB300; fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
WORKLOADS = {"gdn_300m": W.GDN_300M_BF16, "kda_300m": W.KDA_300M_BF16, "gdn_1b": W.GDN_1B_BF16_H0,
             "kda_300m_g16": W.KDA_300M_BF16_G16,
             "mamba2_300m": W.MAMBA2_300M_BF16, "gdn_block_300m": W.GDN_BLOCK_300M_BF16,
             "gdn_tiny": W.GDN_TINY_FP32, "gdn_decode": W.GDN_DECODE_BF16,
             "kda_decode": W.KDA_DECODE_BF16, "gdn_1m": W.GDN_1M_FWD_BF16}
FWD_METRIC = "GDN long-context forward tokens/s on 1 GB300; fraction of roofline"
DECODE_METRIC = "GDN/KDA single-token decode step tokens/s on 1 GB300; fraction of roofline"
BLOCK_METRIC = ("GDN layer token-mixing path (short conv + mixer + gated norm) fwd+bwd tokens/s "
                "on 1 GB300; fraction of roofline")


# ------------------------------------------------------------------ algorithmic work

def algorithmic(w):
    """Per token-head algorithmic FLOPs and bytes of forward and backward.

    FLOPs count the chunk algorithm's own matrix products (forward: decayed
    K K^T, the two WY products, W H, Q H, Q K^T, P U and the state update;
    backward: the recomputed forward products plus the gradient products),
    C^2/3 for the triangular solve; the state recompute is not counted.
    Bytes count each input read once and each output written once."""
    dk, dv, C = w.dk, w.dv, w.chunk
    e = 2 if w.dtype == "bf16" else 4
    sg = (2 if getattr(w, "g_dtype", "f32") == "bf16" else 4) * dk if w.kda else 4
    sb = 4
    fwd_flops = 2 * C * (3 * dk + 2 * dv) + 6 * dk * dv + C * C / 3
    bwd_flops = 2 * C * (7 * dk + 5 * dv) + 14 * dk * dv + C * C / 3
    if not getattr(w, "delta", True):
        # without the delta rule: Q K^T, P U, Q H, the state update (forward);
        # their recompute and the gradient products (backward); no solve
        fwd_flops = 2 * C * (dk + dv) + 4 * dk * dv
        bwd_flops = 2 * C * (2 * dk + 3 * dv) + 8 * dk * dv
    fwd_bytes = e * (2 * dk + 2 * dv) + sg + sb
    bwd_bytes = e * (2 * dk + 2 * dv) + sg + sb + e * (2 * dk + dv) + sg + sb
    return {"fwd_flops": fwd_flops, "bwd_flops": bwd_flops, "fwd_bytes": fwd_bytes,
            "bwd_bytes": bwd_bytes}


def state_bytes(w, kernel):
    """Per-sequence state traffic of a kernel (h0 reads, final state write, dh0)."""
    s = 4 * w.dk * w.dv
    h0 = w.h0_std is not None
    if kernel.endswith("_fwd"):
        return s * (1 + h0)             # ht write (+ h0 read)
    if kernel.endswith("_bwd"):
        return s * (1 + h0)             # dh0 write (+ h0 read in the recompute)
    return 0


def neighbour_bytes(w, kernel):
    """Algorithmic bytes of one launch of a neighbour kernel on workload ``w``:
    each token tensor read once and written once (x -> z; x, dz -> dx; o, gate
    -> out; o, gate, dout -> do, dgate) plus the fp32 weights and their
    gradients; None for other kernels (the partial sums carry none)."""
    e = 2 if w.dtype == "bf16" else 4
    n = w.B * w.T * w.H * w.dk
    taps = w.H * w.dk * w.conv_width * 4
    return {"short_conv_fwd": 2 * e * n + taps, "short_conv_bwd": 3 * e * n + 2 * taps,
            "gated_rmsnorm_fwd": 3 * e * n + 4 * w.dk,
            "gated_rmsnorm_bwd": 5 * e * n + 8 * w.dk}.get(kernel)


def kernel_work(w, kernel):
    """(algorithmic bytes, FLOPs) of one launch of ``kernel`` on workload ``w``.

    The forward kernel carries the forward op's work; the backward op's work
    is carried by its main reverse-scan kernel (the state recompute and the
    partial-sum reduction are implementation overhead and carry none)."""
    nb = neighbour_bytes(w, kernel)
    if nb is not None:
        return float(nb), 0.0
    if kernel == "sum_partials":
        return 0.0, 0.0
    a = algorithmic(w)
    th = w.B * w.T * w.H
    seqs = w.B * w.H
    if kernel.endswith("_fwd"):
        return a["fwd_bytes"] * th + state_bytes(w, kernel) * seqs, a["fwd_flops"] * th
    if kernel.endswith("_bwd"):
        return a["bwd_bytes"] * th + state_bytes(w, kernel) * seqs, a["bwd_flops"] * th
    return 0.0, 0.0


KERNEL_SOURCES = {"tc": "gdn_tc.cu", "simt": "gdn_simt.cu", "decode": "gdn_decode.cu", "kda": "kda_tc.cu"}


def recorded_traffic(kernel, workload_key):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary
    ``profiles/<kernel>_<workload_key>_*.md``, or None when there is none or
    when the kernel source has changed since it was captured."""
    import glob
    import hashlib
    files = glob.glob(os.path.join(ROOT, "profiles", f"{kernel}_{workload_key}*.md"))
    if not files:
        return None
    fields = {}
    for line in open(files[0]):
        if ":" in line and not line.startswith(("|", "#", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().split()[0] if v.strip() else ""
    src = os.path.join(ROOT, "gated_delta_rule_bwd_gb300", "csrc",
                       KERNEL_SOURCES.get(kernel.split("_")[0], ""))
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if sha != fields.get("kernel_source_sha256_16"):
            return None
        return float(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self, t0=None, t1=None):
        """Clock record of the samples taken between wall-clock times t0 and t1
        (the timed region); all samples if none fall inside."""
        import datetime
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 10 and f[2].replace(".", "").isdigit():
                    try:
                        ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        ts = None
                    rows.append([ts] + f[1:])
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [r for r in rows if t0 is not None and r[0] is not None and t0 <= r[0] <= t1]
        in_region = bool(inside)
        rows = inside or rows
        rows = [r[1:] for r in rows]
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = [n for i, n in enumerate(names) if any(r[5 + i].lower() == "active" for r in rows)]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": in_region,
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ------------------------------------------------------------------ CPU oracle timing

def cpu_oracle_run(w, rows, seed=0):
    """Oracle forward + backward over ``rows`` batch rows of workload ``w``."""
    import oracle
    x = w.make(device="cpu", seed=seed, B=rows)
    nthreads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.fwd(x.q, x.k, x.v, x.g, x.beta, x.h0, kda=w.kda, nthreads=nthreads, delta=w.delta)
    if not w.fwd_only:
        oracle.bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, None, kda=w.kda, nthreads=nthreads,
                   delta=w.delta)
    return time.perf_counter() - t0, nthreads


def cpu_baseline(w, min_s=10.0, max_s=30.0):
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    rows = max(1, cores // w.H)
    elapsed, tokens, batches = 0.0, 0, 0
    while elapsed < min_s and (elapsed == 0.0 or elapsed + elapsed / batches <= max_s):
        dt, nthreads = cpu_oracle_run(w, rows, seed=batches)
        elapsed += dt
        tokens += rows * w.T
        batches += 1
    return {"value": tokens / elapsed, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{batches} x ({rows} batch rows x {w.H} heads x {w.T} tokens) of {w.name}, "
                      f"fp64 token recurrence fwd+bwd, {elapsed:.1f} s"}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_tokens_per_s(tokens_per_step, steps, world, slowest_rank_s):
    """Whole-job throughput: every rank processes its own batch (weak scaling),
    timed by the slowest rank."""
    return tokens_per_step * steps * world / slowest_rank_s


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import gated_delta_rule_bwd_gb300 as gdn

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    fwd_s = getattr(gdn, f"{w.mixer}_fwd_save")
    bwd_s = getattr(gdn, f"{w.mixer}_bwd_saved")
    fwd = getattr(gdn, f"{w.mixer}_fwd")
    bwd = getattr(gdn, f"{w.mixer}_bwd")

    x = w.make(device=dev, seed=rank)
    # the training step: the forward keeps the per-chunk entry states and
    # solve results in the saved context, the backward reads them
    ctx = gdn.new_ctx(x.q, x.v, w.chunk, w.kda, w.delta)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        o, ht, _ = fwd_s(x.q, x.k, x.v, x.g, x.beta, x.h0, chunk=w.chunk, ctx=ctx)
        gr = bwd_s(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, ctx, None, chunk=w.chunk)
        return o, ht, gr

    def step_recompute():
        # the same step with the backward recomputing the context (ctx as workspace)
        o, ht = fwd(x.q, x.k, x.v, x.g, x.beta, x.h0, chunk=w.chunk, workspace=ctx)
        gr = bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, None, chunk=w.chunk, workspace=ctx)
        return o, ht, gr

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]

    def timed_steps(fn, cap, n=K):
        # cap = 0: the library only counts its launches (no events between its
        # kernels, which may then overlap one another's start and end)
        with gdn.KernelTimer(cap=cap) as t:
            for i in range(n):
                flush.fill_(i & 0xFF)  # evict L2 between timed steps (outside the events)
                starts[i].record(stream)
                fn()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return ([s.elapsed_time(e) for s, e in zip(starts[:n], ends[:n])], t.launches,
                t.records() if cap else [])

    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(ws)
        torch.cuda.synchronize(dev)
        wall0, epoch0 = time.perf_counter(), time.time()
        step_ms, launches, _ = timed_steps(step, 0)
        wall, epoch1 = time.perf_counter() - wall0, time.time()
        barrier(ws)
    dev_s = sum(step_ms) / 1e3
    dev_s_max = max_over_ranks(dev_s, ws, dev)
    # the same steps again (at most 100 of them) with every library kernel
    # bracketed by events
    _, _, records = timed_steps(step, 64 * min(K, 100), min(K, 100))

    # the recomputing variant of the step, timed the same way (reported beside)
    for _ in range(args.warmup):
        step_recompute()
    rc_ms, _, _ = timed_steps(step_recompute, 0)
    rc_s_max = max_over_ranks(sum(rc_ms) / 1e3, ws, dev)

    # per-kernel live timing (events recorded on the launch stream)
    per = {}
    for name, ms in records:
        per.setdefault(name, []).append(ms)
    totals = {k: sum(v) for k, v in per.items()}
    dom = max(totals, key=totals.get)
    dom_ms = statistics.mean(per[dom])
    peaks, peak_src = load_peaks()
    nbytes, flops = kernel_work(w, dom)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": nbytes / (dom_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (dom_ms * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    wkey = next((k for k, v in WORKLOADS.items() if v is w), w.name)
    roof["traffic"] = args.traffic if args.traffic is not None else recorded_traffic(dom, wkey)
    roof.update({"kernel": dom, "kernel_ms": dom_ms, "peak_source": peak_src,
                 "kernel_timing": "CUDA events around each library kernel on its launch stream, "
                                  "over a second pass of the same K timed steps",
                 "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
                 "kernel_share": totals[dom] / sum(totals.values()),
                 "per_kernel_ms": {k: statistics.mean(v) for k, v in per.items()}})
    # whole-step roofline (every kernel of fwd + bwd against the op's algorithmic work)
    a = algorithmic(w)
    th = w.B * w.T * w.H
    step_bytes = (a["fwd_bytes"] + a["bwd_bytes"]) * th
    step_flops = (a["fwd_flops"] + a["bwd_flops"]) * th
    roof_step_s = max(step_bytes / (peaks["hbm_gbs"] * 1e9), step_flops / (peaks["bf16_tflops"] * 1e12))

    tokens_step = w.B * w.T
    value = aggregate_tokens_per_s(tokens_step, K, ws, dev_s_max)
    ms_step = dev_s_max * 1e3 / K

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(gdn, w, x, ctx, dev, stream, K, args.warmup, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds, 3 * args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "op": w.mixer + " fwd+bwd",
                       "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                       "gate_dtype": "bf16" if w.g_dtype == "bf16" else "f32",
                       "tokens_per_step": tokens_step, "global_batch": w.B * ws,
                       "parallelism": f"replicas x{ws} (independent sequences)",
                       "l2": "flushed between timed steps (2 x L2 buffer written outside the events)",
                       "roofline_step_us": roof_step_s * 1e6,
                       "step_frac_of_roofline": roof_step_s / (ms_step * 1e-3),
                       "wall_s": wall},
            "saved_context": {"bytes": ctx.numel(), "what": "forward keeps each chunk's entry "
                              "state and solve result for the backward"},
            "recompute_variant": {"ms_per_step": rc_s_max * 1e3 / K,
                                  "value": aggregate_tokens_per_s(tokens_step, K, ws, rc_s_max),
                                  "what": "backward recomputes the context (*_fwd + *_bwd)"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches * ws, "clocks": clocks.summary(epoch0, epoch1),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(gdn, w, x, ctx, dev, stream, K, warmup, ws):
    """The mixer step through the public API with pinned host buffers (see
    ``pipelined_e2e``)."""
    fwd_s = getattr(gdn, f"{w.mixer}_fwd_save")
    bwd_s = getattr(gdn, f"{w.mixer}_bwd_saved")
    names = ["q", "k", "v", "g", "beta", "do"] + (["h0"] if x.h0 is not None else [])

    def compute(d):
        o, ht, _ = fwd_s(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("h0"), chunk=w.chunk,
                         ctx=ctx)
        gr = bwd_s(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("h0"), d["do"], ctx, None,
                   chunk=w.chunk)
        return {"o": o, "ht": ht, **{k: v for k, v in gr.items() if v is not None}}

    return pipelined_e2e(names, x, compute, dev, stream, K, warmup, ws, w.B * w.T)


def pipelined_e2e(names, src, compute, dev, stream, K, warmup, ws, tokens_per_step):
    """A step through the public API with pinned host buffers: every step's
    host-to-device copy of its inputs and device-to-host copy of every result
    are inside the timed region.  The loop is pipelined the way a training
    input pipeline is: step i+1's inputs are copied in on one stream and step
    i-1's results copied out on another while step i computes (two sets of
    device input buffers; each result's memory is held until its copy ends).
    ``compute(d)`` runs one step on the device inputs ``d`` (a dict by name)
    and returns its results by name."""
    host_in = {n: getattr(src, n).cpu().pin_memory() for n in names}
    dev_in = [{n: torch.empty_like(getattr(src, n)) for n in names} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    n_copy = 1  # copy streams per direction (two measured no faster: the host link is the limit)
    s_in = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    s_out = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    host_out = {}
    d2h = 0

    def run(n_steps):
        nonlocal d2h
        ready = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]  # inputs copied in
        done = [torch.cuda.Event() for _ in range(2)]    # a buffer set's step finished
        pending = []                                      # results whose copy-out is in flight

        def copy_in(i):
            bi = i % 2
            for j, st in enumerate(s_in):
                with torch.cuda.stream(st):
                    if i >= 2:
                        st.wait_event(done[bi])         # the step that last used this set is done
                    for n in names[j::n_copy]:
                        dev_in[bi][n].copy_(host_in[n], non_blocking=True)
                    ready[bi][j].record(st)

        copy_in(0)
        for i in range(n_steps):
            bi = i % 2
            if i + 1 < n_steps:
                copy_in(i + 1)
            for ev in ready[bi]:
                stream.wait_event(ev)
            outs = compute(dev_in[bi])
            done[bi].record(stream)
            for j, st in enumerate(s_out):
                with torch.cuda.stream(st):
                    st.wait_event(done[bi])
                    for k in list(outs)[j::n_copy]:
                        v = outs[k]
                        if k not in host_out:
                            host_out[k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                        host_out[k].copy_(v, non_blocking=True)
                        v.record_stream(st)
            pending.append(outs)
            if len(pending) > 2:
                pending.pop(0)
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        for st in s_in + s_out:
            stream.wait_stream(st)

    run(max(1, warmup))
    torch.cuda.synchronize(dev)
    barrier(ws)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for st in s_in:
        st.wait_stream(stream)     # the first copy-in starts after t0
    run(K)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    s = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    return {"value": tokens_per_step * K * ws / s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "pipelined": "copy-in of step i+1 and copy-out of step i-1 "
            "overlap step i (one copy stream per direction)"}


# ------------------------------------------------------------------ mixer block

def block_oracle_run(w, rows, seed=0):
    """The oracle's composition of the block (short convolutions, mixer, gated
    norm; forward and backward) over ``rows`` batch rows of workload ``w``."""
    import numpy as np
    import oracle
    from oracle import neighbours as nb
    x = w.make_block(device="cpu", seed=seed, B=rows)
    f = lambda t: t.double().numpy()
    H, D = w.H, w.dk
    shp = (rows, w.T, H, D)
    nthreads = os.cpu_count() or 1
    t0 = time.perf_counter()
    q = nb.short_conv_fwd(f(x.xq), f(x.wq), H, True, D ** -0.5)[0].reshape(shp)
    k = nb.short_conv_fwd(f(x.xk), f(x.wk), H, True, 1.0)[0].reshape(shp)
    v = nb.short_conv_fwd(f(x.xv), f(x.wv), H, False, 1.0)[0].reshape(shp)
    o, _ = oracle.fwd(q, k, v, x.g, x.beta, None, kda=w.kda, nthreads=nthreads)
    nb.gated_rmsnorm_fwd(o, f(x.gate), f(x.weight))
    do, _, _ = nb.gated_rmsnorm_bwd(o, f(x.gate), f(x.weight), f(x.dout))
    gr = oracle.bwd(q, k, v, x.g, x.beta, None, do, None, kda=w.kda, nthreads=nthreads)
    flat = lambda a: np.ascontiguousarray(a).reshape(rows, w.T, H * D)
    nb.short_conv_bwd(f(x.xq), f(x.wq), flat(gr["dq"]), H, True, D ** -0.5)
    nb.short_conv_bwd(f(x.xk), f(x.wk), flat(gr["dk"]), H, True, 1.0)
    nb.short_conv_bwd(f(x.xv), f(x.wv), flat(gr["dv"]), H, False, 1.0)
    return time.perf_counter() - t0, nthreads


def run_block(args):
    """One step = the GDN layer's token-mixing path, forward and backward:
    three short convolutions, the mixer (saved context), the gated norm, then
    the norm's, the mixer's and the convolutions' backward passes."""
    import gated_delta_rule_bwd_gb300 as gdn
    from gated_delta_rule_bwd_gb300.block import block_bwd, block_fwd

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    x = w.make_block(device=dev, seed=rank)
    shp = (w.B, w.T, w.H, w.dk)
    ctx = gdn.new_ctx(x.xq.view(shp), x.xv.view(shp), w.chunk, w.kda)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def compute(d):
        out, ht, saved = block_fwd(d["xq"], d["xk"], d["xv"], d["wq"], d["wk"], d["wv"], d["g"],
                                   d["beta"], d["gate"], d["weight"], chunk=w.chunk, kda=w.kda,
                                   ctx=ctx)
        gr = block_bwd(saved, d["dout"])
        return {"out": out, "ht": ht, **{k: v for k, v in gr.items() if v is not None}}

    dx = {n: getattr(x, n) for n in ("xq", "xk", "xv", "wq", "wk", "wv", "g", "beta", "gate",
                                     "weight", "dout")}

    def step():
        return compute(dx)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]

    def timed_steps(cap, n=K):
        with gdn.KernelTimer(cap=cap) as t:
            for i in range(n):
                flush.fill_(i & 0xFF)  # evict L2 between timed steps (outside the events)
                starts[i].record(stream)
                step()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return [s.elapsed_time(e) for s, e in zip(starts[:n], ends[:n])], t.launches, \
            (t.records() if cap else [])

    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(ws)
        torch.cuda.synchronize(dev)
        epoch0 = time.time()
        step_ms, launches, _ = timed_steps(0)
        epoch1 = time.time()
        barrier(ws)
    dev_s_max = max_over_ranks(sum(step_ms) / 1e3, ws, dev)
    n_ev = min(K, 100)
    _, _, records = timed_steps(64 * n_ev, n_ev)
    per = {}
    for name, ms in records:
        per.setdefault(name, []).append(ms)
    totals = {k: sum(v) for k, v in per.items()}
    peaks, peak_src = load_peaks()
    dom = max(totals, key=totals.get)
    dom_ms = statistics.mean(per[dom])
    nbytes, flops = kernel_work(w, dom)
    roof = {"bound": "hbm", "achieved": nbytes / (dom_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "kernel": dom, "kernel_ms": dom_ms, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
            "kernel_share": totals[dom] / sum(totals.values()),
            "kernel_timing": f"CUDA events around each library kernel on its launch stream, "
                             f"over {n_ev} more steps",
            "per_kernel_ms": {k: statistics.mean(v) for k, v in per.items()},
            "launches_per_step": {k: len(v) / n_ev for k, v in per.items()}}
    roof["frac"] = roof["achieved"] / roof["peak"]
    wkey = next((k for k, v in WORKLOADS.items() if v is w), w.name)
    roof["traffic"] = args.traffic if args.traffic is not None else recorded_traffic(dom, wkey)
    # each neighbour kernel against its own bytes
    nbr = {}
    for k, v in per.items():
        b = neighbour_bytes(w, k)
        if b is not None:
            m = statistics.mean(v)
            nbr[k] = {"ms": m, "achieved_gbs": b / (m * 1e-3) / 1e9,
                      "frac": b / (m * 1e-3) / 1e9 / peaks["hbm_gbs"], "bytes": b}
    roof["neighbour_kernels"] = nbr
    # whole-step roofline: the mixer's work plus every neighbour launch's bytes
    a = algorithmic(w)
    th = w.B * w.T * w.H
    step_bytes = (a["fwd_bytes"] + a["bwd_bytes"]) * th + sum(
        neighbour_bytes(w, k) * len(v) / n_ev for k, v in per.items()
        if neighbour_bytes(w, k) is not None)
    step_flops = (a["fwd_flops"] + a["bwd_flops"]) * th
    roof_step_s = max(step_bytes / (peaks["hbm_gbs"] * 1e9),
                      step_flops / (peaks["bf16_tflops"] * 1e12))
    ms_step = dev_s_max * 1e3 / K
    tokens_step = w.B * w.T

    e2e = None
    if not args.no_e2e:
        e2e = pipelined_e2e(list(dx), x, compute, dev, stream, K, args.warmup, ws, tokens_step)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows, elapsed, batches = 1, 0.0, 0
        while elapsed < args.cpu_seconds:
            dt, nthreads = block_oracle_run(w, rows, seed=batches)
            elapsed += dt
            batches += 1
        cpu = {"value": rows * w.T * batches / elapsed, "unit": "tokens/s", "cores": nthreads,
               "kind": "oracle", "sample": f"{batches} x ({rows} batch row x {w.H} heads x {w.T} "
               f"tokens) of {w.name}: fp64 convolutions, token recurrence and norm, fwd+bwd, "
               f"{elapsed:.1f} s"}

    if rank == 0:
        line = {
            "metric": BLOCK_METRIC, "value": aggregate_tokens_per_s(tokens_step, K, ws, dev_s_max),
            "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "op": w.mixer + " block fwd+bwd",
                       "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                       "conv_width": w.conv_width, "tokens_per_step": tokens_step,
                       "parallelism": f"replicas x{ws} (independent sequences)",
                       "l2": "flushed between timed steps (2 x L2 buffer written outside the events)",
                       "roofline_step_us": roof_step_s * 1e6,
                       "step_frac_of_roofline": roof_step_s / (ms_step * 1e-3)},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches * ws, "clocks": clocks.summary(epoch0, epoch1),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ decode

def decode_bytes(w):
    """Algorithmic bytes of one decode call per (b, h): the fp32 state read and
    written once, each token's q, k, v, o and its gate and beta."""
    e = 2 if w.dtype == "bf16" else 4
    sg = 4 * w.dk if w.kda else 4
    return 2 * 4 * w.dk * w.dv + w.T * (e * (2 * w.dk + 2 * w.dv) + sg + 4)


def run_decode(args):
    """One step = one decode call (T tokens for each of B sequences x H heads),
    the states resident and updated in place.  The states exceed the L2, so no
    flush is needed between steps."""
    import gated_delta_rule_bwd_gb300 as gdn

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    dec = gdn.kda_decode if w.kda else gdn.gdn_decode
    x = w.make(device=dev, seed=rank)
    state = x.h0.clone()
    stream = torch.cuda.current_stream(dev)

    def step():
        return dec(x.q, x.k, x.v, x.g, x.beta, state)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(ws)
        torch.cuda.synchronize(dev)
        epoch0 = time.time()
        with gdn.KernelTimer(cap=0) as counter:
            t0.record(stream)
            for _ in range(K):
                step()
            t1.record(stream)
        torch.cuda.synchronize(dev)
        epoch1 = time.time()
        barrier(ws)
    dev_s_max = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    n_ev = min(K, 200)
    with gdn.KernelTimer(cap=2 * n_ev) as timer:
        for _ in range(n_ev):
            step()
    torch.cuda.synchronize(dev)
    per = [ms for name, ms in timer.records() if name == "decode"]
    kern_ms = statistics.mean(per)
    peaks, peak_src = load_peaks()
    nbytes = decode_bytes(w) * w.B * w.H
    roof = {"bound": "hbm", "achieved": nbytes / (kern_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "kernel": "decode", "kernel_ms": kern_ms, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": nbytes,
            "kernel_timing": f"CUDA events around each of {n_ev} launches on the launch stream"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    wkey = next((k for k, v in WORKLOADS.items() if v is w), w.name)
    roof["traffic"] = args.traffic if args.traffic is not None else recorded_traffic("decode", wkey)

    e2e = None
    if not args.no_e2e:
        # per step: this step's q, k, v, g, beta in from pinned host memory and
        # its o out (the states stay on the device, as in serving)
        names = ["q", "k", "v", "g", "beta"]
        host = {n: getattr(x, n).cpu().pin_memory() for n in names}
        o_host = torch.empty((w.B, w.T, w.H, w.dv), dtype=x.q.dtype, pin_memory=True)
        dbuf = {n: torch.empty_like(getattr(x, n)) for n in names}

        def e2e_step():
            for n in names:
                dbuf[n].copy_(host[n], non_blocking=True)
            o, _ = dec(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"], state)
            o_host.copy_(o, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        es = max_over_ranks(e0.elapsed_time(e1) / 1e3, ws, dev)
        e2e = {"value": w.B * w.T * K * ws / es, "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
               "d2h_bytes_per_step": o_host.numel() * o_host.element_size()}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        rows = max(1, (os.cpu_count() or 1) // w.H)
        xs = w.make(device="cpu", seed=0, B=rows)
        oracle.fwd(xs.q, xs.k, xs.v, xs.g, xs.beta, xs.h0, kda=w.kda)  # warm
        c0, n = time.perf_counter(), 0
        while time.perf_counter() - c0 < args.cpu_seconds:
            oracle.fwd(xs.q, xs.k, xs.v, xs.g, xs.beta, xs.h0, kda=w.kda)
            n += 1
        dt = time.perf_counter() - c0
        cpu = {"value": rows * w.T * n / dt, "unit": "tokens/s", "cores": os.cpu_count() or 1,
               "kind": "oracle", "sample": f"{n} x ({rows} sequences x {w.H} heads x {w.T} token) "
               f"of {w.name}, fp64 token recurrence, {dt:.1f} s"}

    if rank == 0:
        ms_step = dev_s_max * 1e3 / K
        line = {
            "metric": DECODE_METRIC, "value": w.B * w.T * K * ws / dev_s_max, "unit": "tokens/s",
            "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "op": ("kda" if w.kda else "gdn") + " decode",
                       "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                       "tokens_per_step": w.B * w.T, "parallelism": f"replicas x{ws}",
                       "l2": "not flushed: the states (fp32) exceed the L2",
                       "state_bytes": w.B * w.H * w.dk * w.dv * 4},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": counter.launches * ws, "clocks": clocks.summary(epoch0, epoch1),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ forward only

def run_forward(args):
    """One step = one forward call over the whole workload (the 1M-token
    context: the tensor-core forward runs each sequence in segments).  The
    inputs (12 GB of bf16 q, k, v) exceed the L2, so no flush is needed."""
    import gated_delta_rule_bwd_gb300 as gdn

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    fwd = gdn.kda_fwd if w.kda else gdn.gdn_fwd
    x = w.make(device=dev, seed=rank)
    wsb = torch.empty(max(16, gdn.fwd_workspace_bytes(x.q, x.v, w.chunk, w.kda)),
                      dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return fwd(x.q, x.k, x.v, x.g, x.beta, x.h0, chunk=w.chunk, workspace=wsb)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(ws)
        torch.cuda.synchronize(dev)
        epoch0 = time.time()
        with gdn.KernelTimer(cap=0) as counter:
            t0.record(stream)
            for _ in range(K):
                step()
            t1.record(stream)
        torch.cuda.synchronize(dev)
        epoch1 = time.time()
        barrier(ws)
    dev_s_max = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    n_ev = min(K, 5)
    with gdn.KernelTimer(cap=16 * n_ev) as timer:
        for _ in range(n_ev):
            step()
    torch.cuda.synchronize(dev)
    per = {}
    for name, ms in timer.records():
        per.setdefault(name, []).append(ms)
    totals = {k: sum(v) for k, v in per.items()}
    dom = max(totals, key=totals.get)
    peaks, peak_src = load_peaks()
    a = algorithmic(w)
    th = w.B * w.T * w.H
    nbytes = a["fwd_bytes"] * th + state_bytes(w, "tc_fwd") * w.B * w.H
    ms_step = dev_s_max * 1e3 / K
    # the op's algorithmic bytes against the whole call (solve, segment passes,
    # combine and output pass together)
    roof = {"bound": "hbm", "achieved": nbytes / (ms_step * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "kernel": "whole forward call", "peak_source": peak_src,
            "algorithmic_bytes_per_launch": nbytes, "traffic": None,
            "per_kernel_ms_per_call": {k: v / n_ev for k, v in totals.items()},
            "dominant_kernel": dom,
            "kernel_timing": f"CUDA events around each library kernel over {n_ev} calls"}
    roof["frac"] = roof["achieved"] / roof["peak"]

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        Ts = 1 << 14  # a bounded sample: every head, the first 16384 tokens
        xs = w.make(device="cpu", seed=0, T=Ts)
        c0, n = time.perf_counter(), 0
        while n == 0 or time.perf_counter() - c0 < args.cpu_seconds:
            oracle.fwd(xs.q, xs.k, xs.v, xs.g, xs.beta, xs.h0, kda=w.kda)
            n += 1
        dt = time.perf_counter() - c0
        cpu = {"value": w.B * Ts * n / dt, "unit": "tokens/s", "cores": os.cpu_count() or 1,
               "kind": "oracle", "sample": f"{n} x ({w.B} x {Ts} tokens x {w.H} heads) of "
               f"{w.name}, fp64 token recurrence, forward, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": FWD_METRIC, "value": w.B * w.T * K * ws / dev_s_max, "unit": "tokens/s",
            "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "op": ("kda" if w.kda else "gdn") + " fwd",
                       "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                       "tokens_per_step": w.B * w.T, "parallelism": f"replicas x{ws}",
                       "l2": "not flushed: the inputs exceed the L2"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": None,
            "gpu_launches": counter.launches * ws, "clocks": clocks.summary(epoch0, epoch1),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    rows = max(1, cores // w.H)
    run = block_oracle_run if w.block else cpu_oracle_run
    if w.block:
        rows = 1
    for i in range(args.warmup):
        run(w, rows, seed=1000 + i)
    times = []
    nthreads = cores
    for i in range(args.steps):
        dt, nthreads = run(w, rows, seed=i)
        times.append(dt)
    total = sum(times)
    value = rows * w.T * args.steps / total
    sample = (f"each step: {rows} batch rows x {w.H} heads x {w.T} tokens of {w.name} "
              f"(fp64 token recurrence fwd+bwd on {nthreads} threads"
              + ("; with the fp64 short convolutions and gated norm)" if w.block else ")"))
    line = {"impl": "reference", "metric": BLOCK_METRIC if w.block else METRIC, "value": value,
            "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "op": w.mixer + (" block" if w.block else "") + " fwd+bwd",
                       "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: 1000 timed steps (about 0.6 s at the 300M shape, long enough for
    # clock samples inside the timed region) for this library, 20 for the CPU
    # oracle (about 0.3 s a step)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gdn_300m")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    decode = wl.T == 1 and wl.fwd_only
    fwd_only = wl.fwd_only and not decode
    if args.steps is None:
        # the 1M-token forward takes about 18 ms a step
        ours = 5000 if decode else 40 if fwd_only else 1000
        args.steps = 20 if args.impl == "reference" else ours
    if args.warmup is None:
        args.warmup = 3 if args.impl == "reference" or args.steps < 100 else 20
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        if decode or fwd_only:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                              "training step; this workload has its CPU oracle timing in "
                              "cpu_baseline"}))
            return
        run_reference(args)
    elif wl.block:
        run_block(args)
    elif decode:
        run_decode(args)
    elif fwd_only:
        run_forward(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
