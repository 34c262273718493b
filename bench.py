"""Benchmark: attention forward TFLOP/s on GB300, and its fraction of the dense
FP16/BF16 tensor peak, across the sequence lengths of the isolated-attention
benchmark of the noflash-attention forum post (ai-navigate-news, section "It's
actually faster too!": B=1, H=16, D=64, fp16, non-causal, N = 256 ... 16384).

One step = one forward launch per sequence length of the sweep on synthetic
seeded inputs already resident in HBM.  Every launch is timed with CUDA events
on the launching stream; before each launch, outside the timed events, L2 is
flushed by a 256 MiB write followed by a 256 MiB read of a second buffer, so
the inputs are not in L2 and the launch does not pay for writing back the
flush's own dirty lines (the state ncu's cache control gives).  Each sequence
length's time is the median of its launches over the timed steps; value =
sum of algorithmic FLOPs / sum of those times.  The default run also times,
in the same region and with their own events, the head-dim-128 points of the
>= 60%-of-peak target (video-DiT at N = 17600 and 75600, the training forward
at N = 8192) under "d128", the backward of the training and GQA-prefill
workloads under "bwd", and the GQA causal prefill forward (N = 1024 .. 16384)
under "gqa_prefill_fwd".  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config sweep|gqa_prefill|video_dit|training|tiny|gqa_decode]

--config gqa_decode times the split-key forward (attn_fwd_splitkv) on decode
shapes and reports GB/s against the HBM copy bandwidth instead of TFLOP/s.

--impl reference times the fp64 CPU oracle (the reference arm) on the host
cores: each step is a bounded sample of the same workload.  Under torchrun
(N > 1) every rank runs its own replica (the path needs no exchange); rank 0
prints the line, with value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense FP16/BF16 tensor peak vs seq len"
METRIC_BWD = "attention bwd TFLOP/s on 1 GB300 (5 products of the forward's size, halved for causal)"
METRIC_DECODE = ("attention decode GB/s on 1 GB300 (split-key forward against a KV cache: "
                 "Q, K, V read once, O and LSE written)")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "fwd_traffic.json")


def peaks():
    """Measured denominators from MEASURED_PEAKS.json when it exists, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = x
            walk(d)

            def find(*keys):
                for k, v in flat.items():
                    kl = k.lower()
                    if all(s in kl for s in keys) and isinstance(v, (int, float)):
                        return float(v)
                return None
            sus = find("bf16", "sustain")
            burst = None
            for k, v in flat.items():
                kl = k.lower()
                if "bf16" in kl and "sustain" not in kl and isinstance(v, (int, float)) and v > 100:
                    burst = float(v)
                    break
            hbm = find("hbm")
            if burst:
                return {"bf16_tflops": burst, "bf16_tflops_sustained": sus or burst,
                        "hbm_gbs": hbm or FALLBACK_PEAKS["hbm_gbs"], "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash() -> str:
    """Hash of the forward kernel's code with comments and blank space
    removed: an edit of a comment leaves the recorded traffic valid, any
    change of code voids it."""
    import re
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "ptx.cuh", "bias.cuh", "splitkv.cu", "vconv.cu"):
        with open(os.path.join(ROOT, "tiled_memory_efficient_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def traffic_for(workload: str, n: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    try:
        d = json.load(open(PROFILE_TRAFFIC))
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("per_launch_dram_bytes", {}).get(f"{workload}:{n}")


class L2Flush:
    """Evicts the inputs from L2 between timed launches: a 256 MiB write
    (larger than the 129 MB L2) and then a 256 MiB read of another buffer,
    which writes the dirty lines back before the timed region starts."""
    NOTE = "flushed before every launch (256 MiB write + 256 MiB read, outside the timed events)"

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, flops_per_rank: float, slowest_ms: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (slowest_ms * 1e-3) / 1e12


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return dist, dist.get_rank(), world, local
    if n_gpus != 1:
        raise SystemExit("--gpus N > 1 must be launched with torchrun (one rank per GPU)")
    return None, 0, 1, 0


def run_ours(args):
    import torch

    from tiled_memory_efficient_gb300 import _lib, inputs

    dist, rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS[args.config]
    seq = list(w.seq_lens) if args.n is None else [args.n]
    _lib.load()
    pk = peaks()
    stream = torch.cuda.current_stream(dev)

    bwd = args.pass_ == "bwd"
    decode = w.nq is not None
    if decode and bwd:
        raise SystemExit("the decode workload has no backward pass")
    splits = {n: _lib.num_splits(w.B, w.Hq, w.Hkv, w.queries(n), n, w.D) for n in seq}
    # the unmasked forward goes through attn_fwd_ws (its workspace allocated
    # here, outside the timed region); --plain times attn_fwd
    use_ws = not (args.plain or bwd or decode or args.mask != "none")
    ws_splits = {n: _lib.fwd_ws_splits(w.B, w.Hq, w.Hkv, n, n, w.D, w.causal) if use_ws else 1
                 for n in seq}
    if args.mask != "none" and decode:
        raise SystemExit("--mask is for the prefill / training workloads")
    # inputs resident in HBM before the timed region
    bufs = []
    for n in seq:
        x = inputs.make_inputs(w, n)
        if bwd and "do" not in x:
            g = torch.Generator().manual_seed(inputs.seed_for(w, n) + 1)
            x["do"] = torch.randn(x["q"].shape, generator=g).to(w.dtype)
        q, k, v = (x[m].to(dev) for m in ("q", "k", "v"))
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
        extra = None
        x["mask"] = make_bench_mask(args.mask, w, n, dev)
        if bwd:
            _lib.attn_fwd(q, k, v, causal=w.causal, out=out, lse=lse, mask=x["mask"])
            do = x["do"].to(dev)
            ws = torch.empty(max(16, _lib.load().attn_bwd_workspace_size(
                w.B, w.Hq, w.Hkv, n, n, w.D, 1 if w.dtype == torch.bfloat16 else 0)),
                device=dev, dtype=torch.uint8)
            extra = (do, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), ws)
        elif decode:
            extra = torch.empty(max(16, _lib.splitkv_workspace_size(
                w.B, w.Hq, w.Hkv, w.queries(n), n, w.D, splits[n])), device=dev, dtype=torch.uint8)
        elif use_ws:
            extra = torch.empty(max(16, _lib.fwd_workspace_size(w.B, w.Hq, w.Hkv, n, n, w.D,
                                                               w.dtype)),
                                device=dev, dtype=torch.uint8)
        bufs.append((n, q, k, v, out, lse, x, extra))
    # The head-dim-128 points of the >= 60%-of-peak target (video-DiT at
    # N = 17600 and 75600, the training forward at N = 8192), timed in the
    # same region as the sweep with their own events; reported under "d128".
    d128 = []
    bwdp = []
    gqap = []
    if (args.config == "sweep" and not bwd and args.mask == "none" and args.n is None
            and not args.no_d128):
        for name, n in GQA_POINTS:
            wd = inputs.WORKLOADS[name]
            x = inputs.make_inputs(wd, n)
            q, k, v = (x[m].to(dev) for m in ("q", "k", "v"))
            ws = torch.empty(max(16, _lib.fwd_workspace_size(wd.B, wd.Hq, wd.Hkv, n, n, wd.D,
                                                             wd.dtype)),
                             device=dev, dtype=torch.uint8)
            gqap.append((wd, n, q, k, v, torch.empty_like(q),
                         torch.empty(q.shape[:3], device=dev, dtype=torch.float32), ws))
            del x
        for name, n in D128_POINTS:
            wd = inputs.WORKLOADS[name]
            x = inputs.make_inputs(wd, n)
            q, k, v = (x[m].to(dev) for m in ("q", "k", "v"))
            ws = torch.empty(max(16, _lib.fwd_workspace_size(wd.B, wd.Hq, wd.Hkv, n, n, wd.D,
                                                             wd.dtype)),
                             device=dev, dtype=torch.uint8)
            d128.append((wd, n, q, k, v, torch.empty_like(q),
                         torch.empty(q.shape[:3], device=dev, dtype=torch.float32), ws))
            del x
        # the backward of the training workload and of GQA prefill (attn_bwd,
        # with the workspace attn_bwd_workspace_size recommends)
        for name, n in BWD_POINTS:
            wd = inputs.WORKLOADS[name]
            x = inputs.make_inputs(wd, n)
            if "do" not in x:
                g = torch.Generator().manual_seed(inputs.seed_for(wd, n) + 1)
                x["do"] = torch.randn(x["q"].shape, generator=g).to(wd.dtype)
            q, k, v, do = (x[m].to(dev) for m in ("q", "k", "v", "do"))
            out, lse = _lib.attn_fwd(q, k, v, causal=wd.causal)
            ws = torch.empty(max(16, _lib.load().attn_bwd_workspace_size(
                wd.B, wd.Hq, wd.Hkv, n, n, wd.D, 1 if wd.dtype == torch.bfloat16 else 0)),
                device=dev, dtype=torch.uint8)
            bwdp.append((wd, n, q, k, v, out, lse, do, torch.empty_like(q), torch.empty_like(k),
                         torch.empty_like(v), ws))
            del x
    flush = L2Flush(dev)

    def launch(b):
        n, q, k, v, out, lse, x, extra = b
        if bwd:
            do, dq, dk, dv, ws = extra
            _lib.attn_bwd(q, k, v, out, do, lse, causal=w.causal, dq=dq, dk=dk, dv=dv,
                          workspace=ws, mask=x["mask"])
        elif decode:
            _lib.attn_fwd_splitkv(q, k, v, causal=w.causal, splits=splits[n], out=out, lse=lse,
                                  workspace=extra)
        elif use_ws:
            _lib.attn_fwd_ws(q, k, v, causal=w.causal, out=out, lse=lse, workspace=extra)
        else:
            _lib.attn_fwd(q, k, v, causal=w.causal, out=out, lse=lse, mask=x["mask"])

    def launch_d128(b, plain=False):
        wd, n, q, k, v, out, lse, ws = b
        if plain:   # attn_fwd: the value tiles are converted inside every CTA
            _lib.attn_fwd(q, k, v, causal=wd.causal, out=out, lse=lse)
        else:       # attn_fwd_ws: converted once per call into the workspace (timed with it)
            _lib.attn_fwd_ws(q, k, v, causal=wd.causal, out=out, lse=lse, workspace=ws)

    def launch_bwdp(b):
        wd, n, q, k, v, out, lse, do, dq, dk, dv, ws = b
        _lib.attn_bwd(q, k, v, out, do, lse, causal=wd.causal, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(args.warmup):
        for b in bufs:
            flush()
            launch(b)
        for b in bwdp:
            flush()
            launch_bwdp(b)
        for b in d128:
            flush()
            launch_d128(b)
            flush()
            launch_d128(b, plain=True)
        for b in gqap:
            flush()
            launch_d128(b)
    rc = _lib.sync_status(dev)
    if rc != _lib.ATTN_OK:
        raise RuntimeError(f"device status after warm-up: {_lib.strerror(rc)}")

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in bufs] for _ in range(args.steps)]
    ev_d = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in d128] for _ in range(args.steps)]
    ev_p = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in d128] for _ in range(args.steps)]
    ev_b = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in bwdp] for _ in range(args.steps)]
    ev_g = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in gqap] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_wall = time.perf_counter()
        for s in range(args.steps):
            for i, b in enumerate(bufs):
                flush()
                ev[s][i][0].record(stream)
                launch(b)
                ev[s][i][1].record(stream)
            for i, b in enumerate(bwdp):
                flush()
                ev_b[s][i][0].record(stream)
                launch_bwdp(b)
                ev_b[s][i][1].record(stream)
            for i, b in enumerate(d128):
                flush()
                ev_d[s][i][0].record(stream)
                launch_d128(b)
                ev_d[s][i][1].record(stream)
                flush()
                ev_p[s][i][0].record(stream)
                launch_d128(b, plain=True)
                ev_p[s][i][1].record(stream)
            for i, b in enumerate(gqap):
                flush()
                ev_g[s][i][0].record(stream)
                launch_d128(b)
                ev_g[s][i][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    rc = _lib.sync_status(dev)
    if rc != _lib.ATTN_OK:
        raise RuntimeError(f"device status after timing: {_lib.strerror(rc)}")

    per_launch_ms = [[ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
                     for i in range(len(bufs))]
    # per sequence length: the median launch time over the timed steps
    ms_each = [statistics.median(x) for x in per_launch_ms]
    # backward: 5 products of the forward's size (S recomputed, dP, dV, dK, dQ);
    # decode: algorithmic bytes instead of FLOPs (the work is HBM-bound)
    flops = [(2.5 if bwd else 1.0) * w.flops_fwd(n) for n in seq]
    work = [w.bytes_fwd(n) for n in seq] if decode else flops
    scale = 1e9 if decode else 1e12
    unit = "GB/s" if decode else "TFLOP/s"
    step_ms = max_over_ranks(sum(ms_each), dist, dev)
    value = world * sum(work) / (step_ms * 1e-3) / scale

    # roofline of the dominant launch (largest share of the step time)
    dom = max(range(len(seq)), key=lambda i: ms_each[i])
    achieved = work[dom] / (ms_each[dom] * 1e-3) / scale
    peak = pk["hbm_gbs"] if decode else pk["bf16_tflops"]
    traffic = traffic_for(args.config, seq[dom]) if (use_ws or decode or bwd) else None
    if bwd:
        traffic = None
    if decode:
        kernel = ("attn_fwd_kernel over key ranges + splitkv_merge_kernel (one call)"
                  if splits[seq[dom]] > 1 else "attn_fwd_kernel")
        peak_source = f"{pk['source']} HBM copy bandwidth"
    else:
        kernel = ("attn_bwd (stats + dK/dV + dQ kernels)" if bwd else
                  "attn_fwd_kernel" if not use_ws else
                  "attn_fwd_ws: " + ("v_to_f16_kernel + " if w.dtype == torch.bfloat16 else "") +
                  "attn_fwd_kernel" + (" + splitkv_merge_kernel" if ws_splits[seq[dom]] > 1 else ""))
        peak_source = f"{pk['source']} bf16 dense (burst; fp16 runs at the same tensor rate)"
    roofline = {"bound": "hbm" if decode else "tensor", "achieved": round(achieved, 1),
                "peak": peak, "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": kernel, "launch": f"N={seq[dom]}", "peak_source": peak_source}

    # end to end through the public call with host buffers: H2D of q,k,v from
    # pinned memory, the forward, D2H of out and lse, every step
    # (decode: the KV cache lives on the device, as in serving; only the new
    # queries go up and the outputs come back)
    e2e = None
    if not args.no_e2e and not bwd:
        host = []
        h2d = d2h = 0
        for n, q, k, v, out, lse, x, _ in bufs:
            hq, hk, hv = (x[m].pin_memory() for m in ("q", "k", "v"))
            ho = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
            hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
            host.append((hq, hk, hv, ho, hl))
            h2d += sum(t.numel() * t.element_size() for t in ((hq,) if decode else (hq, hk, hv)))
            d2h += ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e_steps = max(1, min(args.steps, 10))
        # Copies overlap the kernels (decode excepted): inputs go up on one stream, outputs come
        # back on another, the kernels run on the compute stream; events order
        # every reuse of a buffer (its upload waits for the previous step's
        # kernel on it, the kernel for the previous download of its outputs).
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        nb = len(bufs)
        h2d_done = [torch.cuda.Event() for _ in range(nb)]
        k_done = [torch.cuda.Event() for _ in range(nb)]
        d2h_done = [torch.cuda.Event() for _ in range(nb)]
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        for step in range(e2e_steps):
            for i, (b, (hq, hk, hv, ho, hl)) in enumerate(zip(bufs, host)):
                n, q, k, v, out, lse = b[:6]
                if decode:
                    # a few KB each way: cross-stream events would cost more
                    # than they hide, so everything stays on one stream
                    q.copy_(hq, non_blocking=True)
                    launch(b)
                    ho.copy_(out, non_blocking=True)
                    hl.copy_(lse, non_blocking=True)
                    continue
                with torch.cuda.stream(up):
                    if step > 0:
                        up.wait_event(k_done[i])
                    q.copy_(hq, non_blocking=True)
                    k.copy_(hk, non_blocking=True)
                    v.copy_(hv, non_blocking=True)
                    h2d_done[i].record(up)
                stream.wait_event(h2d_done[i])
                if step > 0:
                    stream.wait_event(d2h_done[i])
                launch(b)
                k_done[i].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(k_done[i])
                    ho.copy_(out, non_blocking=True)
                    hl.copy_(lse, non_blocking=True)
                    d2h_done[i].record(down)
        stream.wait_stream(down)
        stream.wait_stream(up)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
        e2e = {"value": round(world * sum(work) / (e2e_ms * 1e-3) / scale, 2), "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}

    clocks = clk.summary()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None if (args.no_cpu_baseline or world > 1 or bwd or args.mask != "none") else \
        cpu_baseline(w, seq, budget_s=args.cpu_budget)
    if decode:
        sweep = [{"Nk": n, "ms": round(ms, 4), "splits": splits[n],
                  "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                  "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
                 for n, ms, b in zip(seq, ms_each, work)]
    else:
        sweep = [{"N": n, "ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1),
                  "frac_of_peak": round(f / (ms * 1e-3) / 1e12 / peak, 4)}
                 for n, ms, f in zip(seq, ms_each, flops)]
    def fwd_launches(wd, n, ws_call):
        if not ws_call:
            return 1
        return (1 + (wd.dtype == torch.bfloat16) +
                (_lib.fwd_ws_splits(wd.B, wd.Hq, wd.Hkv, n, n, wd.D, wd.causal) > 1))

    def bwd_launches(wd, n):
        return 3 + (_lib.bwd_splits(wd.B, wd.Hq, wd.Hkv, n, n, wd.D, wd.causal) > 1)

    launches_per_step = (
        sum((2 if splits[n] > 1 else 1) if decode else bwd_launches(w, n) if bwd else
            fwd_launches(w, n, use_ws) for n in seq) +
        sum(fwd_launches(wd, n, True) + 1 for wd, n, *_ in d128) +
        sum(fwd_launches(wd, n, True) for wd, n, *_ in gqap) +
        sum(bwd_launches(wd, n) for wd, n, *_ in bwdp))
    bwd_rep = None
    if bwdp:
        pts = []
        for i, (wd, n, *_rest) in enumerate(bwdp):
            ms = statistics.median(ev_b[s_][i][0].elapsed_time(ev_b[s_][i][1])
                                   for s_ in range(args.steps))
            tf = 2.5 * wd.flops_fwd(n) / (ms * 1e-3) / 1e12
            pts.append({"workload": wd.note, "N": n, "ms": round(ms, 4), "tflops": round(tf, 1),
                        "frac_of_peak": round(tf / pk["bf16_tflops"], 4)})
        bwd_rep = {"entry": "attn_bwd (statistics, dQ, dK/dV kernels, each a programmatic "
                            "dependent of the one before; dK/dV partial sums and their "
                            "reduction when the dK/dV grid is cut into query ranges)",
                   "flops": "5 products of the forward's size (2.5 x the forward's "
                            "4*B*Hq*Nq*Nk*D, halved under the causal mask)",
                   "timing": "median call time over the timed steps, CUDA events, L2 flushed "
                             "before every call", "points": pts}
    d128_rep = None
    if d128:
        pts = []
        for i, (wd, n, *_rest) in enumerate(d128):
            ms = statistics.median(ev_d[s_][i][0].elapsed_time(ev_d[s_][i][1])
                                   for s_ in range(args.steps))
            ms_p = statistics.median(ev_p[s_][i][0].elapsed_time(ev_p[s_][i][1])
                                     for s_ in range(args.steps))
            tf = wd.flops_fwd(n) / (ms * 1e-3) / 1e12
            tf_p = wd.flops_fwd(n) / (ms_p * 1e-3) / 1e12
            pts.append({"workload": wd.note, "N": n, "ms": round(ms, 4), "tflops": round(tf, 1),
                        "frac_of_peak": round(tf / pk["bf16_tflops"], 4),
                        "frac_of_sustained_peak": round(tf / pk["bf16_tflops_sustained"], 4),
                        "attn_fwd_ms": round(ms_p, 4), "attn_fwd_tflops": round(tf_p, 1)})
        d128_rep = {"target": "forward >= 60% of the dense FP16/BF16 tensor peak at N >= 8K, D = 128",
                    "peak": pk["bf16_tflops"], "sustained_peak": pk["bf16_tflops_sustained"],
                    "peak_source": f"{pk['source']} bf16 dense (burst and sustained)",
                    "entry": "attn_fwd_ws: the bf16 value tensor is converted to fp16 once "
                             "per call (a first kernel, included in the time); attn_fwd_*: "
                             "the same forward with the conversion inside every CTA",
                    "timing": "median call time over the timed steps, CUDA events, L2 "
                              "flushed before every call; clocks: the line's clocks record "
                              "(same timed region)",
                    "points": pts,
                    "met": all(p_["frac_of_peak"] >= 0.6 for p_ in pts)}
    gqa_rep = None
    if gqap:
        pts = []
        for i, (wd, n, *_rest) in enumerate(gqap):
            ms = statistics.median(ev_g[s_][i][0].elapsed_time(ev_g[s_][i][1])
                                   for s_ in range(args.steps))
            tf = wd.flops_fwd(n) / (ms * 1e-3) / 1e12
            pts.append({"workload": wd.note, "N": n, "ms": round(ms, 4), "tflops": round(tf, 1),
                        "frac_of_peak": round(tf / pk["bf16_tflops"], 4),
                        "key_ranges": _lib.fwd_ws_splits(wd.B, wd.Hq, wd.Hkv, n, n, wd.D,
                                                         wd.causal),
                        "half_positions": _lib.fwd_half_positions(wd.B, wd.Hq, wd.Hkv, n, n,
                                                                  wd.D, wd.causal, wd.dtype)})
        gqa_rep = {"entry": "attn_fwd_ws (causal FLOPs: half of 4*B*Hq*N*N*D)",
                   "timing": "median call time over the timed steps, CUDA events, L2 flushed "
                             "before every call", "points": pts}
    metric = METRIC_DECODE if decode else (METRIC_BWD if bwd else METRIC)
    line = {
        "metric": metric, "value": round(value, 2), "unit": unit,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if w.dtype == torch.float16 else "bf16",
        "data": "synthetic",
        "config": bench_config(w, seq, args.mask, world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks, "sweep": sweep, "d128": d128_rep, "bwd": bwd_rep,
        "gqa_prefill_fwd": gqa_rep,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if args.config == "sweep" and not bwd and args.mask == "none":
        line["context"] = {
            "source": "the pages' isolated-attention table (noflash-attention forum post, "
                      "\"It's actually faster too!\"): one AMD MI50 (gfx906, 150 W), FP16, "
                      "the pages' tiled PyTorch-matmul kernel; context only",
            "per_N": [{"N": n, "ms": PAGES_MI50_MS[n],
                       "tflops": round(w.flops_fwd(n) / (PAGES_MI50_MS[n] * 1e-3) / 1e12, 2),
                       "ratio_here": round(PAGES_MI50_MS[n] / ms, 1)}
                      for n, ms in zip(seq, ms_each) if n in PAGES_MI50_MS]}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


D128_POINTS = (("video_dit", 17600), ("video_dit", 75600), ("training", 8192))
# The pages' own timings of this sweep: the noflash-attention forum post
# (ai-navigate-news, section "It's actually faster too!", the isolated
# attention table: B=1, H=16, D=64, FP16 on one AMD MI50 (gfx906) at a 150 W
# limit, the pages' tiled PyTorch-matmul kernel), in ms.  Another machine and
# another implementation: reported as context, never as the target.
PAGES_MI50_MS = {256: 0.18, 512: 0.29, 1024: 0.85, 2048: 4.74, 4096: 17.93, 8192: 72.75,
                 16384: 1325.69}
BWD_POINTS = (("training", 8192), ("gqa_prefill", 4096))
# the GQA causal prefill forward (Hq=14, Hkv=2, D=64 fp16), through attn_fwd_ws
GQA_POINTS = tuple(("gqa_prefill", n) for n in (1024, 2048, 4096, 8192, 16384))


def bench_config(w, seq, mask, world):
    """The config of a bench line: the same dict for both arms."""
    return {"workload": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
            "causal": w.causal, "seq_lens": seq, "Nq": w.nq if w.nq is not None else "= N",
            "mask": MASK_NOTES[mask],
            "inputs": "seeded N(0,1) rounded to dtype" +
                      ("; 1% of key rows x8" if w.outlier_keys else ""),
            "l2": L2Flush.NOTE,
            "parallelism": "replicas" if world > 1 else "single GPU"}


MASK_NOTES = {
    "none": None,
    "padding": "bool key-padding mask [B,1,1,N] keeping the first 7N/8 keys; FLOPs counted "
               "unmasked (every key tile is still visited)",
    "additive": "additive N(0,1) bias [1,1,N,N] in the input dtype",
}


def make_bench_mask(kind, w, n, dev):
    """The attn_mask of a masked measurement (None for unmasked runs)."""
    import torch
    if kind == "none":
        return None
    if kind == "padding":
        return (torch.arange(n, device=dev) < n - n // 8).reshape(1, 1, 1, n).expand(
            w.B, 1, 1, n).contiguous()
    g = torch.Generator().manual_seed(inputs_seed_for_mask(n))
    return torch.randn((1, 1, n, n), generator=g).to(w.dtype).to(dev)


def inputs_seed_for_mask(n: int) -> int:
    return 77_000 + n


def cpu_baseline(w, seq, budget_s: float = 15.0, n_override=None):
    """The fp64 oracle, as it stands, on the host cores: a sample of query rows
    (spread over the heads of batch 0; every batch for decode shapes) of the
    largest sequence length, sized to about `budget_s` seconds.  Decode shapes
    report GB/s: the sampled rows' share of the workload's algorithmic bytes."""
    import numpy as np

    import oracle
    from tiled_memory_efficient_gb300 import inputs
    n = n_override or max(seq)
    nq = w.queries(n)
    decode = w.nq is not None
    threads = oracle.default_threads()
    x = inputs.make_inputs(w, n)
    nb = w.B if decode else 1
    q, k, v = x["q"][:nb], x["k"][:nb], x["v"][:nb]
    total_rows = nb * w.Hq * nq

    def flops_rows(rows):
        keys = sum(oracle.attended_keys(int(r) % nq, n, w.causal, nq) for r in rows)
        return 4.0 * w.D * keys

    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(total_rows, size=min(total_rows, 8 * threads), replace=False))
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, causal=w.causal, rows=probe, threads=threads)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    for _ in range(3):  # re-size from the last run until it fills about the budget
        n_rows = int(min(total_rows, max(len(probe), budget_s / per_row)))
        rows = np.sort(rng.choice(total_rows, size=n_rows, replace=False))
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, causal=w.causal, rows=rows, threads=threads)
        dt = time.perf_counter() - t0
        per_row = dt / n_rows
        if dt >= 0.5 * budget_s or n_rows == total_rows:
            break
    if decode:
        value, unit = n_rows / (w.B * w.Hq * nq) * w.bytes_fwd(n) / dt / 1e9, "GB/s"
        where = f"all {w.B} sequences, Nk={n}"
    else:
        value, unit = flops_rows(rows) / dt / 1e12, "TFLOP/s"
        where = f"batch 0 at N={n}"
    return {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{n_rows} of the {total_rows} query rows of {where} (seeded, all heads; "
                      f"each row over its visible keys{', causal ' + str(w.causal) if w.causal else ''}),"
                      f" fp64, {dt:.3f} s"}


def run_reference(args):
    """Reference arm: the fp64 oracle on the host cores, bounded sample per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    from tiled_memory_efficient_gb300 import inputs
    w = inputs.WORKLOADS[args.config]
    seq = list(w.seq_lens) if args.n is None else [args.n]
    decode = w.nq is not None
    threads = oracle.default_threads()
    data = {}
    for n in seq:
        x = inputs.make_inputs(w, n)
        data[n] = (x["q"][:1, :1], x["k"][:1, :1], x["v"][:1, :1])
    nqs = {n: w.queries(n) for n in seq}
    # rows per N per step, sized so the whole run takes about --ref-seconds
    budget_step = max(0.05, args.ref_seconds / (args.steps + args.warmup))
    cost = {n: 4.0 * w.D * n for n in seq}          # flops per full row
    tot = sum(cost.values())
    rng = np.random.default_rng(0)
    # calibrate
    t0 = time.perf_counter()
    q, k, v = data[seq[-1]]
    cal = rng.choice(nqs[seq[-1]], size=min(nqs[seq[-1]], 4 * threads), replace=False)
    oracle.attention_fwd(q, k, v, causal=w.causal, rows=cal, threads=threads)
    rate = cost[seq[-1]] * len(cal) / max(time.perf_counter() - t0, 1e-4)   # flops/s
    rows_per_n = {n: max(1, min(nqs[n], int(budget_step * rate * (cost[n] / tot) / cost[n])))
                  for n in seq}
    step_work = 0.0
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        fl = 0.0
        for n in seq:
            q, k, v = data[n]
            rows = rng.choice(nqs[n], size=rows_per_n[n], replace=False)
            oracle.attention_fwd(q, k, v, causal=w.causal, rows=rows, threads=threads)
            if decode:   # the rows' share of the workload's algorithmic bytes
                fl += len(rows) / (w.B * w.Hq * nqs[n]) * w.bytes_fwd(n)
            else:
                fl += sum(4.0 * w.D * oracle.attended_keys(int(i), n, w.causal, nqs[n])
                          for i in rows)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
            step_work += fl
    total = sum(times)
    value = step_work / total / (1e9 if decode else 1e12)
    unit = "GB/s" if decode else "TFLOP/s"
    sample = (f"per step: rows {rows_per_n} of head (b=0,h=0) per N, all visible keys, fp64 "
              f"({threads} threads)")
    line = {
        "metric": METRIC_DECODE if decode else METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / max(1, len(times)), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": bench_config(w, seq, args.mask, world),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


FFN_CONFIG = {"workload": "token-chunked SwiGLU FFN of the Qwen 2.5 0.5B shape (d_model 896, "
                          "d_ff 4864, no biases), bf16, 16384 tokens in chunks of 4096",
              "T": 16384, "d_model": 896, "d_ff": 4864, "act": "swiglu", "chunk": 4096}
METRIC_FFN = "token-chunked FFN TFLOP/s on 1 GB300 (both products, 3 d_model x d_ff GEMMs per token)"


def ffn_host_inputs():
    """The FFN workload's seeded host tensors (bf16): x, W1 = [Wg; Wu], W2."""
    import torch
    c = FFN_CONFIG
    T, d, f = c["T"], c["d_model"], c["d_ff"]
    g = torch.Generator().manual_seed(9000)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w1 = (torch.randn(2 * f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return x, w1, w2


def ffn_oracle_sample(x, w1, w2, budget_s: float, seed: int = 0):
    """Times the fp64 FFN oracle on seeded row samples of x for about
    budget_s seconds.  Returns (TFLOP/s, rows per call, calls, cores, seconds)."""
    import numpy as np
    import torch

    from oracle import ffn as ffn_oracle
    c = FFN_CONFIG
    d, f = c["d_model"], c["d_ff"]
    rng = np.random.default_rng(seed)
    rows = 64
    w1d, w2d = w1.double().numpy(), w2.double().numpy()
    calls, flops, t_all = 0, 0.0, 0.0
    while t_all < budget_s:
        idx = rng.choice(x.shape[0], size=rows, replace=False)
        xs = x[idx].double().numpy()
        t0 = time.perf_counter()
        ffn_oracle.ffn_fwd(xs, w1d, None, w2d, None, c["act"], h_dtype=torch.bfloat16)
        t_all += time.perf_counter() - t0
        flops += 2.0 * rows * d * 2 * f + 2.0 * rows * f * d
        calls += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return flops / t_all / 1e12, rows, calls, cores, t_all


def run_reference_ffn(args):
    """Reference arm of --config ffn: the fp64 FFN oracle (numpy matrix
    products and the activations) on the host cores, a bounded row sample of
    the same workload per step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    x, w1, w2 = ffn_host_inputs()
    per_step = max(0.2, args.ref_seconds / (args.steps + args.warmup))
    ffn_oracle_sample(x, w1, w2, per_step * args.warmup, seed=1)
    tf, rows, calls, cores, secs = ffn_oracle_sample(x, w1, w2, per_step * args.steps, seed=2)
    sample = f"{calls} calls of {rows} seeded token rows each, fp64 (numpy BLAS)"
    print(json.dumps({
        "metric": METRIC_FFN, "value": round(tf, 6), "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference", "config": FFN_CONFIG,
        "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_ffn(args):
    """--config ffn: the chunked FFN (include/ffn.h), one step = one forward
    over T tokens; FLOPs = 2 T d_model (2 d_ff) + 2 T d_ff d_model."""
    import torch

    from tiled_memory_efficient_gb300 import _lib
    dist, rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    c = FFN_CONFIG
    T, d, f = c["T"], c["d_model"], c["d_ff"]
    hx, hw1, hw2 = ffn_host_inputs()
    x, w1, w2 = hx.to(dev), hw1.to(dev), hw2.to(dev)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    lib = _lib.load()
    ws = torch.empty(lib.ffn_workspace_size(T, f, c["chunk"]), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    flops = 2.0 * T * d * 2 * f + 2.0 * T * f * d

    def step():
        _lib.ffn_forward(x, w1, None, w2, None, act=c["act"], chunk=c["chunk"], out=y, workspace=ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(dev.index or 0) as clk:
        for e0, e1 in ev:
            flush()
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
    rc = _lib.sync_status(dev)
    if rc != _lib.ATTN_OK:
        raise RuntimeError(f"device status after timing: {_lib.strerror(rc)}")
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    ms = max_over_ranks(ms, dist, dev)
    pk = peaks()
    tf = flops / (ms * 1e-3) / 1e12
    n_chunks = (T + c["chunk"] - 1) // c["chunk"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ctf, rows, calls, cores, _ = ffn_oracle_sample(hx, hw1, hw2, args.cpu_budget)
        cpu = {"value": round(ctf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{calls} calls of {rows} seeded token rows each, fp64 (numpy BLAS)"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC_FFN, "value": round(world * tf, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(c, l2=L2Flush.NOTE.replace("launch", "step")),
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / pk["bf16_tflops"], 4),
                         "traffic": None, "kernel": "ffn_gemm_kernel (both products, all chunks)",
                         "peak_source": f"{pk['source']} bf16 dense (burst)"},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps * 2 * n_chunks,
            "clocks": clk.summary()}), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="sweep")
    ap.add_argument("--n", type=int, default=None, help="run one sequence length only")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--plain", action="store_true",
                    help="time attn_fwd instead of attn_fwd_ws (the default for unmasked "
                         "forwards: bf16 value tiles converted once per call into a workspace, "
                         "unevenly filled grids cut into key ranges)")
    ap.add_argument("--no-d128", action="store_true",
                    help="leave the head-dim-128 target points out of the default sweep run")
    ap.add_argument("--mask", choices=["none", "padding", "additive"], default="none",
                    help="time the masked kernels with this attn_mask")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the cpu_baseline of a GPU run")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="seconds of oracle time for a whole --impl reference run")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.config == "ffn":
        if args.impl == "reference":
            run_reference_ffn(args)
            return
        run_ffn(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
