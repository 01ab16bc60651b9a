#!/usr/bin/env python3
"""Benchmark of the Simple GLA hot path on one GB300 (or N replicas).

One step = one chunked prefill forward over the Laplace-3B-shaped layer
(B8 T2048 H16 dk96 dv192, chunk 128, bf16) and one recurrent decode step over
N1280 x H16 states (fp32 96x192), both through libgla's C ABI with inputs
resident in HBM.  The K timed steps run as two phases (K prefills, then K
decodes) so that neither kernel is charged for the other's write-backs.  ``value`` is prefill tokens/s (tokens of the layer,
all 16 heads, per second of prefill time, summed over replicas); the decode
half is reported as state GB/s under ``decode``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 the script runs under torchrun, one replica per GPU (weak scaling,
no data-path collective); timing is the max over ranks.  ``--impl reference``
times the fp64 CPU reference on the host instead (rank 0 only).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GLA fwd tokens/s (H16,dk96,dv192,bf16) + %TC peak; decode state GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def prefill_bytes(B, T, H, dk, dv, with_h0, with_hT):
    """Algorithmic HBM bytes of one prefill launch: bf16 q, k, v read, bf16 out written, f32 states."""
    per_token_head = 2 * (dk + dk + dv + dv)
    b = B * T * H * per_token_head
    st = B * H * dk * dv * 4
    return b + (st if with_h0 else 0) + (st if with_hT else 0)


def prefill_flops(B, T, H, dk, dv, C):
    """Tensor-core FLOPs issued per launch as full tiles: 2C(dk+dv) + 4 dk dv per token-head."""
    return B * T * H * (2 * C * (dk + dv) + 4 * dk * dv)


def backward_flops(B, T, H, dk, dv, C):
    """Tensor-core FLOPs of the chunked backward per launch, as full tiles (chunk C = 128): per chunk the
    scores K Q^T, V dO^T, dO V^T and dV = P dO + K G, dK = P Q + V G^T, dQ = P K + dO S^T, plus the
    chunk recurrence of the gradient state G (dk x dv per token).  Per token-head:
    6 C (dk + dv) + 6 dk dv + 2 dk dv.  The forward state S_{c-1} recomputed by this implementation
    (one more state pass, 2 x 128 x dv issued per token-head, M padded to 128) is not counted."""
    return B * T * H * (6 * C * (dk + dv) + 8 * dk * dv)


def backward_bytes(B, T, H, dk, dv, nseq=None, with_h0=False, with_dhT=False, with_dh0=True):
    """The method's HBM bytes per gla_chunk_bwd launch: read q, k, v and dout (bf16), write dq, dk, dv
    (bf16): 2 (2 dk + 2 dv) + 2 (2 dk + dv) bytes per token-head, 1,920 at dk 96, dv 192; plus the f32
    states (h0, dhT in; dh0 out) per chain."""
    nseq = B if nseq is None else nseq
    st = nseq * H * dk * dv * 4
    return (B * T * H * (2 * (2 * dk + 2 * dv) + 2 * (2 * dk + dv)) + (st if with_h0 else 0) +
            (st if with_dhT else 0) + (st if with_dh0 else 0))


def backward_impl_bytes(B, T, H, dk, dv, C=128):
    """HBM bytes this implementation moves per gla_chunk_bwd launch beyond the method's own: the two state
    passes read k, v and q, dout once more (2 (2 dk + 2 dv) per token-head), and the bf16 images of the
    states S_{c-1} and G_c are written once and read once (8 dk dv / C per token-head)."""
    return B * T * H * (2 * (2 * dk + 2 * dv) + 8 * dk * dv // C)


# Datasheet HBM3e bandwidth of one GB300 (about 8 TB/s): the denominator of the decode fractions.  The
# measured copy bandwidth (a torch tensor copy) is reported next to it; a streaming kernel such as the
# decode step can run above that copy.
HBM_NOMINAL_GBS = 8000.0


def decode_bytes(N, H, dk, dv):
    state = N * H * dk * dv * 4 * 2
    io = N * H * (2 * dk + 2 * dv) * 2
    return state, io


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        finally:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, x in enumerate(r) if x.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel_source, key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[key]
        if d.get("source_sha") == source_hash(kernel_source):
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def dist_setup(init: bool = True):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and init:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------------
_REF_INPUTS = {}


def reference_inputs():
    """The layer workload on the host (seed 0), widened once to the reference's float32 input format."""
    if not _REF_INPUTS:
        from gated_linear_rnn_gb300 import inputs as I
        w = I.WORKLOADS["layer_bf16"]
        d = I.make_prefill(w, device="cpu", seed=0)
        _REF_INPUTS.update({k: d[k].float().numpy() for k in ("q", "k", "v")})
        _REF_INPUTS["log_decay"] = d["log_decay"].double().numpy()
        _REF_INPUTS["w"] = w
    return _REF_INPUTS


def reference_pass(row: int, threads: int) -> float:
    """The fp64 reference over one batch row of the layer (all H heads, T tokens); returns seconds."""
    import oracle
    d = reference_inputs()
    sl = slice(row, row + 1)
    t0 = time.perf_counter()
    oracle.recurrent(d["q"][sl], d["k"][sl], d["v"][sl], d["log_decay"], None, nthreads=threads)
    return time.perf_counter() - t0


def cpu_reference_rate(budget_s: float):
    """fp64 reference (as it stands) on the host cores over rows of the layer workload, for about
    ``budget_s`` seconds; returns (tokens/s, threads, sample description)."""
    import oracle
    d = reference_inputs()
    w = d["w"]
    threads = oracle.default_threads()
    el, rows = 0.0, 0
    while el < budget_s or rows == 0:
        el += reference_pass(rows % w.B, threads)
        rows += 1
    sample = (f"{rows} batch row(s) of the layer workload (each: {w.H} heads x T={w.T}), "
              f"{el:.1f} s of fp64 reference time")
    return rows * w.T / el, threads, sample


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    d = reference_inputs()
    w = d["w"]
    threads = oracle.default_threads()
    times = []
    for i in range(args.warmup + args.steps):
        t = reference_pass(i % w.B, threads)
        if i >= args.warmup:
            times.append(t)
    tot = sum(times)
    value = len(times) * w.T / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: the fp64 reference over one batch row ({w.H} heads x T={w.T})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": "Laplace-3B-shaped GLA layer prefill B8 T2048 H16 dk96 dv192 chunk128 bf16 "
                        "+ decode step N1280 x H16 (fp32 state 96x192)",
            "global_batch": w.B, "seq_len": w.T, "heads": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
            "decode_sequences": 1280,
            "l2": "inputs larger than L2 every iteration (302 MB prefill io, 1.51 GB decode state); no flush"}


def run_ours(args, world, rank, local):
    import torch

    from gated_linear_rnn_gb300 import build as Bld
    from gated_linear_rnn_gb300 import gla
    from gated_linear_rnn_gb300 import inputs as I

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Bld.build_library()
    gla.load()
    peaks, peak_src = load_peaks()

    w = I.WORKLOADS["layer_bf16"]
    wd = I.WORKLOADS["decode"]
    P = I.make_prefill(w, device=dev, seed=rank)
    D = I.make_decode(wd, device=dev, seed=rank)
    B, T, H, dk, dv, C = w.B, w.T, w.H, w.dk, w.dv, w.chunk
    out = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    dout = torch.empty(wd.B, wd.H, wd.dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def prefill():
        gla.gla_chunk_fwd(P["q"], P["k"], P["v"], P["log_decay"], P["h0"], out, hT, C, None, stream)

    def decode():
        gla.gla_decode_step(D["q"], D["k"], D["v"], D["log_decay"], D["state"], dout, stream)

    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize()
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after warm-up: {st_code} ({gla.gla_status_str(st_code)})")

    # K steps, timed as two back-to-back phases (K prefill launches, then K decode launches) so
    # neither kernel pays for the other's dirty L2 lines; every launch has its own event pair.
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    launches0 = gla.gla_kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            evp[i][0].record(stream)
            prefill()
            evp[i][1].record(stream)
        for i in range(args.steps):
            evd[i][0].record(stream)
            decode()
            evd[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    launches = gla.gla_kernel_launches() - launches0
    pre_ms = [evp[i][0].elapsed_time(evp[i][1]) for i in range(args.steps)]
    dec_ms = [evd[i][0].elapsed_time(evd[i][1]) for i in range(args.steps)]
    pre_total = max_over_ranks(sum(pre_ms), world)
    dec_total = max_over_ranks(sum(dec_ms), world)
    step_total = max_over_ranks(sum(pre_ms) + sum(dec_ms), world)
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the timed region: {st_code} ({gla.gla_status_str(st_code)})")

    tokens = B * T * args.steps * world
    value = tokens / (pre_total / 1e3)
    pbytes = prefill_bytes(B, T, H, dk, dv, P["h0"] is not None, True)
    pflops = prefill_flops(B, T, H, dk, dv, C)
    pre_avg_s = pre_total / args.steps / 1e3
    achieved_gbs = pbytes / pre_avg_s / 1e9
    tc_tflops = pflops / pre_avg_s / 1e12
    tc_kernel = os.path.join(ROOT, "gated_linear_rnn_gb300", "csrc", "gla_tc.cu")
    sbytes, iobytes = decode_bytes(wd.B, wd.H, wd.dk, wd.dv)
    dec_avg_s = dec_total / args.steps / 1e3

    # ---- the other prefill workloads: long context (segmented schedule) and the ragged packed batch ----
    long_leg = run_prefill_workload(args, "long_bf16", stream, peaks, peak_src, dev, rank)
    ragged_leg = run_prefill_workload(args, "ragged", stream, peaks, peak_src, dev, rank)
    tiny_leg = run_tiny_f32(args, stream, dev, rank)

    # ---- end to end through the public API: pinned host inputs in, results back to the host ----
    e2e = run_e2e(args, P, D, w, wd, out, hT, dout, stream)

    # ---- paged decode: the same step through a slot table (a permutation of the state pages) ----
    paged = run_paged_decode(args, D, wd, dout, stream, peaks)

    # ---- the layer prefill with the output gate fused into its epilogue ----
    gated = run_gated_prefill(args, P, w, out, hT, stream, peaks)

    # ---- decode over pages holding all 24 layers of a sequence ----
    layers = run_decode_layers(args, wd, stream, peaks, dev)

    # ---- causal conv1d + SiLU over the layer's residual stream, and its per-token step ----
    conv = run_conv(args, w, wd, stream, peaks, dev)

    # ---- backward of the layer prefill (training path), timed on its own after the step ----
    bwd = run_backward(args, P, w, stream, peaks, peak_src) if args.bwd_steps > 0 else None
    train = run_train_step(args, P, w, stream) if args.bwd_steps > 0 else None

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "prefill_ms": pre_total / args.steps, "decode_ms": dec_total / args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": recorded_traffic(tc_kernel, "prefill_layer_bf16"),
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "kernel": "gla_chunk_fwd (layer_bf16)",
                     "algorithmic_bytes_per_launch": pbytes,
                     "tensor": {"achieved_tflops": tc_tflops, "peak_tflops": peaks["bf16_tflops"],
                                "frac": tc_tflops / peaks["bf16_tflops"],
                                "flops_per_launch": pflops, "peak_source": f"{peak_src} bf16 dense (burst)"}},
        "decode": {"value": sbytes / dec_avg_s / 1e9, "unit": "state GB/s",
                   "total_gbs": (sbytes + iobytes) / dec_avg_s / 1e9,
                   "frac_of_hbm_peak": (sbytes + iobytes) / dec_avg_s / 1e9 / HBM_NOMINAL_GBS,
                   "hbm_peak_gbs": HBM_NOMINAL_GBS, "hbm_peak_source": "GB300 datasheet HBM3e (about 8 TB/s)",
                   "frac_of_measured_copy": (sbytes + iobytes) / dec_avg_s / 1e9 / peaks["hbm_gbs"],
                   "us_per_step": dec_avg_s * 1e6, "state_bytes": sbytes, "io_bytes": iobytes,
                   "tokens_per_s": wd.B * world / dec_avg_s},
        "e2e": e2e,
        "prefill_long": long_leg,
        "prefill_ragged": ragged_leg,
        "prefill_tiny_f32": tiny_leg,
        "decode_paged": paged,
        "prefill_gated": gated,
        "decode_layers": layers,
        "conv1d_silu": conv,
        "backward": bwd,
        "train_step": train,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, sample = cpu_reference_rate(args.cpu_budget)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_prefill_workload(args, name, stream, peaks, peak_src, dev, seed):
    """gla_chunk_fwd on another prefill workload of the pages: ``long_bf16`` (B1 T32768 H16 with h0, the
    segmented schedule) or ``ragged`` (64 packed sequences of U[1, 8192] tokens with per-sequence h0,
    walked longest first).  CUDA events around every launch on the launching stream; inputs are larger
    than L2 (no flush).  Algorithmic bytes: q, k, v read and out written once (1,152 B per token-head at
    dk 96, dv 192) plus the f32 h0 read and hT written per chain."""
    import torch
    from gated_linear_rnn_gb300 import gla
    from gated_linear_rnn_gb300 import inputs as I
    w = I.WORKLOADS[name]
    d = I.make_prefill(w, device=dev, seed=seed)
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].to(dev)
    nseq = d["q"].shape[0] if cu is None else cu.numel() - 1
    rows = d["q"].shape[0] * d["q"].shape[1]
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device=dev)
    hT = torch.empty(nseq, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def step():
        gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, w.chunk, cu, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, min(args.steps, 30))
    l0 = gla.gla_kernel_launches()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for e in ev:
        e[0].record(stream)
        step()
        e[1].record(stream)
    torch.cuda.synchronize()
    launches = (gla.gla_kernel_launches() - l0) // n
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the {name} prefill: {st_code} ({gla.gla_status_str(st_code)})")
    times = [e[0].elapsed_time(e[1]) for e in ev]
    us = statistics.mean(times) * 1e3
    st_bytes = nseq * w.H * w.dk * w.dv * 4
    by = rows * w.H * 2 * (2 * w.dk + 2 * w.dv) + (st_bytes if d["h0"] is not None else 0) + st_bytes
    fl = prefill_flops(1, rows, w.H, w.dk, w.dv, w.chunk)
    gbs = by / (us / 1e6) / 1e9
    e2e = None
    if cu is None:
        # the same forward through the public API on pinned host arrays (gla_chunk_fwd_host; few long
        # sequences are cut into chunk-aligned time ranges so that copies and compute overlap)
        host = {k: d[k].cpu().pin_memory() for k in ("q", "k", "v", "log_decay")}
        h_h0 = None if d["h0"] is None else d["h0"].cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_hT = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()

        def host_step():
            gla.gla_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_decay"], h_h0, h_out, h_hT, w.chunk,
                                   stream)

        for _ in range(2):
            host_step()
        torch.cuda.synchronize()
        ne = max(3, min(args.steps, 8))
        eve = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(ne)]
        for e in eve:
            e[0].record(stream)
            host_step()
            e[1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(e[0].elapsed_time(e[1]) for e in eve)
        h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + [h_h0] if t is not None)
        d2h = h_out.numel() * h_out.element_size() + h_hT.numel() * h_hT.element_size()
        e2e = {"value": rows / (ms / 1e3), "unit": "tokens/s", "ms": ms, "steps": ne, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "copy_gbs": (h2d + d2h) / (ms / 1e3) / 1e9,
               "note": "gla_chunk_fwd_host on pinned host arrays in and out, CUDA events around each call (median)"}
        del host, h_h0, h_out, h_hT
    return {"value": rows / (us / 1e6), "unit": "tokens/s", "us": us, "us_median": statistics.median(times) * 1e3,
            "us_best": min(times) * 1e3, "steps": n, "launches_per_call": launches, "tokens": rows, "sequences": nseq,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": by,
                         "traffic": recorded_traffic(os.path.join(ROOT, "gated_linear_rnn_gb300", "csrc", "gla_tc.cu"),
                                                     f"prefill_{name}"),
                         "tensor": {"achieved_tflops": fl / (us / 1e6) / 1e12, "peak_tflops": peaks["bf16_tflops"],
                                    "frac": fl / (us / 1e6) / 1e12 / peaks["bf16_tflops"], "flops_per_launch": fl}},
            "workload": w.note, "kernel": f"gla_chunk_fwd ({name})", "e2e": e2e}


def run_tiny_f32(args, stream, dev, seed):
    """gla_chunk_fwd_f32 on the small fp32 parity workload (B1 H2 T256 dk=dv=64, chunk 64): CUDA events
    around each of up to 30 back-to-back calls (median).  A latency number, not a roofline one: two chains
    of four chunks occupy two SMs for a few microseconds."""
    import torch
    from gated_linear_rnn_gb300 import gla
    from gated_linear_rnn_gb300 import inputs as I
    w = I.WORKLOADS["tiny_f32"]
    d = I.make_prefill(w, device=dev, seed=seed)
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.float32, device=dev)
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def step():
        gla.gla_chunk_fwd_f32(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, w.chunk, None, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, min(args.steps, 30))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for e in ev:
        e[0].record(stream)
        step()
        e[1].record(stream)
    torch.cuda.synchronize()
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the tiny f32 prefill: {st_code} ({gla.gla_status_str(st_code)})")
    us = statistics.median(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    kind = gla.gla_chunk_kernel(gla.OP_FORWARD, gla.F32, w.dk, w.dv, w.chunk)
    return {"value": w.B * w.T / (us / 1e6), "unit": "tokens/s", "us": us, "steps": n,
            "kernel": "tensor cores" if kind == gla.KERNEL_TENSOR_CORE else "SIMT",
            "workload": w.note, "note": "the parity configuration; latency-bound, reported for completeness"}


def run_paged_decode(args, D, wd, dout, stream, peaks):
    """gla_decode_step_paged over the decode workload's states as a pool, rows in a seeded random
    page order; CUDA events per launch, median."""
    import torch
    from gated_linear_rnn_gb300 import gla
    g = torch.Generator().manual_seed(7)
    slots = torch.randperm(wd.B, generator=g).to(torch.int32).to(D["q"].device)

    def step():
        gla.gla_decode_step_paged(D["q"], D["k"], D["v"], D["log_decay"], D["state"], slots, dout, stream)

    for _ in range(3):
        step()
    n = max(3, min(args.steps, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for e in ev:
        e[0].record(stream)
        step()
        e[1].record(stream)
    torch.cuda.synchronize()
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the paged decode: {st_code} ({gla.gla_status_str(st_code)})")
    us = statistics.median(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    sbytes, iobytes = decode_bytes(wd.B, wd.H, wd.dk, wd.dv)
    iobytes += wd.B * 4  # the slot table
    gbs = (sbytes + iobytes) / (us / 1e6) / 1e9
    return {"us_per_step": us, "unit": "state GB/s", "value": sbytes / (us / 1e6) / 1e9,
            "frac_of_hbm_peak": gbs / HBM_NOMINAL_GBS, "frac_of_measured_copy": gbs / peaks["hbm_gbs"], "steps": n,
            "rows": wd.B, "pool_pages": wd.B}


def run_gated_prefill(args, P, w, out, hT, stream, peaks):
    """gla_chunk_fwd_gated on the layer workload (SiLU gate, g seeded like the output): the output gate
    fused into the forward's epilogue; CUDA events per launch, median.  Algorithmic bytes add one bf16
    read of g per output element to the plain forward's."""
    import torch
    from gated_linear_rnn_gb300 import gla, inputs as I
    g = I.make_gate(out.shape, device=out.device, seed=5)
    C = w.chunk

    def step():
        gla.gla_chunk_fwd_gated(P["q"], P["k"], P["v"], g, P["log_decay"], P["h0"], out, hT, C, None,
                                gate_kind=gla.GATE_SILU, stream=stream)

    for _ in range(3):
        step()
    n = max(3, min(args.steps, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for e in ev:
        e[0].record(stream)
        step()
        e[1].record(stream)
    torch.cuda.synchronize()
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the gated prefill: {st_code} ({gla.gla_status_str(st_code)})")
    us = statistics.median(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    nbytes = prefill_bytes(w.B, w.T, w.H, w.dk, w.dv, P["h0"] is not None, True) + w.B * w.T * w.H * w.dv * 2
    return {"us": us, "unit": "tokens/s", "value": w.B * w.T / (us / 1e6), "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / (us / 1e6) / 1e9, "frac_of_hbm_peak": nbytes / (us / 1e6) / 1e9 / peaks["hbm_gbs"],
            "steps": n, "gate": "silu", "kernel": "gla_chunk_fwd_gated (layer_bf16)"}


def run_decode_layers(args, wd, stream, peaks, dev, N=128, L=24):
    """gla_decode_step_layers: N sequences whose pages hold all L layers (the 24-layer model), one
    launch for every layer, and the same step as L one-layer launches; CUDA events, median."""
    import torch
    from gated_linear_rnn_gb300 import gla, inputs as I
    H, dk, dv = wd.H, wd.dk, wd.dv
    g = torch.Generator(device=dev).manual_seed(13)
    q = (torch.randn(L, N, H, dk, generator=g, device=dev) / dk ** 0.5).to(torch.bfloat16)
    k = (torch.randn(L, N, H, dk, generator=g, device=dev) / dk ** 0.5).to(torch.bfloat16)
    v = torch.randn(L, N, H, dv, generator=g, device=dev).to(torch.bfloat16)
    ld = torch.stack([I.log_decays(H, wd.decay_lo, wd.decay_hi)] * L).to(dev)
    pool = torch.randn(N, L, H, dk, dv, generator=g, device=dev).mul_(0.02)
    slots = torch.randperm(N, device="cpu", generator=torch.Generator().manual_seed(13)).to(torch.int32).to(dev)
    out = torch.empty(L, N, H, dv, dtype=torch.bfloat16, device=dev)

    def one():
        gla.gla_decode_step_layers(q, k, v, ld, pool, slots, out, stream=stream)

    def per_layer():
        for l in range(L):
            gla.gla_decode_step_layers(q[l:l + 1], k[l:l + 1], v[l:l + 1], ld[l:l + 1], pool, slots, out[l:l + 1],
                                       layer0=l, stream=stream)

    res = {}
    for name, fn in (("one_launch", one), ("per_layer", per_layer)):
        for _ in range(3):
            fn()
        n = max(3, min(args.steps, 30))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for e in ev:
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the multi-layer decode: {st_code} ({gla.gla_status_str(st_code)})")
    sbytes, iobytes = decode_bytes(N * L, H, dk, dv)
    us = res["one_launch"]
    gbs = (sbytes + iobytes) / (us / 1e6) / 1e9
    return {"us_one_launch": us, "us_per_layer_launches": res["per_layer"], "unit": "state GB/s",
            "value": sbytes / (us / 1e6) / 1e9, "frac_of_hbm_peak": gbs / HBM_NOMINAL_GBS,
            "frac_of_measured_copy": gbs / peaks["hbm_gbs"],
            "sequences": N, "layers": L, "pool_bytes": pool.numel() * 4}


def run_conv(args, w, wd, stream, peaks, dev, D=3072):
    """gla_conv1d_silu over [B, T, D] bf16 (the layer's residual stream, D = 3072) and
    gla_conv1d_silu_step over [N, D] with the decode workload's N; CUDA events, median."""
    import torch
    from gated_linear_rnn_gb300 import gla
    g = torch.Generator(device=dev).manual_seed(11)
    x = torch.randn(w.B, w.T, D, generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty_like(x)
    wt = torch.randn(D, 4, generator=g, device=dev) * 0.5
    bias = torch.randn(D, generator=g, device=dev) * 0.1
    so = torch.empty(w.B, D, 3, device=dev)
    xs = torch.randn(wd.B, D, generator=g, device=dev).to(torch.bfloat16)
    ys = torch.empty_like(xs)
    st = torch.zeros(wd.B, D, 3, device=dev)

    def timed(fn, n):
        for _ in range(3):
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for e in ev:
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        return statistics.median(e[0].elapsed_time(e[1]) for e in ev)

    n = max(3, min(args.steps, 50))
    ms = timed(lambda: gla.gla_conv1d_silu(x, wt, bias, None, so, y, None, stream), n)
    ms_step = timed(lambda: gla.gla_conv1d_silu_step(xs, wt, bias, st, ys, stream), n)
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the conv: {st_code} ({gla.gla_status_str(st_code)})")
    by = w.B * w.T * D * 2 * 2 + D * 4 * 4 + D * 4 + w.B * D * 3 * 4
    by_step = wd.B * D * 2 * 2 + wd.B * D * 3 * 4 * 2
    return {"value": w.B * w.T / (ms / 1e3), "unit": "tokens/s", "us": ms * 1e3, "shape": [w.B, w.T, D],
            "roofline": {"bound": "hbm", "achieved": by / (ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": by},
            "step": {"us": ms_step * 1e3, "rows": wd.B, "gbs": by_step / (ms_step / 1e3) / 1e9,
                     "frac_of_hbm_peak": by_step / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"]}}


def run_backward(args, P, w, stream, peaks, peak_src):
    """gla_chunk_bwd on the layer workload (h0 = 0, dhT = 0, dout ~ N(0, 1)); CUDA events per call."""
    import torch
    from gated_linear_rnn_gb300 import gla
    g = torch.Generator(device=P["q"].device).manual_seed(1000003)
    do = torch.randn(P["v"].shape, generator=g, device=P["q"].device).to(torch.bfloat16)
    dq, dk_, dv_ = (torch.empty_like(P[k]) for k in ("q", "k", "v"))
    dh0 = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=P["q"].device)

    def step():
        gla.gla_chunk_bwd(P["q"], P["k"], P["v"], do, P["log_decay"], None, None, dq, dk_, dv_, dh0, w.chunk,
                          None, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    l0 = gla.gla_kernel_launches()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.bwd_steps)]
    for e in ev:
        e[0].record(stream)
        step()
        e[1].record(stream)
    torch.cuda.synchronize()
    launches = (gla.gla_kernel_launches() - l0) // max(1, args.bwd_steps)
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the backward: {st_code} ({gla.gla_status_str(st_code)})")
    ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    fl = backward_flops(w.B, w.T, w.H, w.dk, w.dv, w.chunk)
    by = backward_bytes(w.B, w.T, w.H, w.dk, w.dv)
    impl = backward_impl_bytes(w.B, w.T, w.H, w.dk, w.dv, w.chunk)
    gbs = by / (ms / 1e3) / 1e9
    tfl = fl / (ms / 1e3) / 1e12
    return {"value": w.B * w.T / (ms / 1e3), "unit": "tokens/s", "ms": ms, "launches_per_call": launches,
            "steps": args.bwd_steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": by,
                         "algorithmic_bytes_note": "q, k, v, dout read and dq, dk, dv written once (bf16): "
                                                   "1,920 B per token-head, plus dh0",
                         "implementation_extra_bytes_per_launch": impl,
                         "moved_gbs_incl_implementation": (by + impl) / (ms / 1e3) / 1e9,
                         "tensor": {"achieved_tflops": tfl, "peak_tflops": peaks["bf16_tflops"],
                                    "frac": tfl / peaks["bf16_tflops"], "flops_per_launch": fl}},
            "kernel": "gla_chunk_bwd (layer_bf16): two tensor-core state passes + chunk-parallel gradient kernel"}


def run_train_step(args, P, w, stream):
    """One training step of the layer (forward, then backward from dout ~ N(0, 1)) two ways: the plain
    pair gla_chunk_fwd + gla_chunk_bwd, and gla_chunk_fwd_save + gla_chunk_bwd_saved, where the backward
    takes the states the forward left instead of walking the chains again.  CUDA events per step."""
    import torch
    from gated_linear_rnn_gb300 import gla
    g = torch.Generator(device=P["q"].device).manual_seed(1000003)
    do = torch.randn(P["v"].shape, generator=g, device=P["q"].device).to(torch.bfloat16)
    out = torch.empty_like(do)
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=P["q"].device)
    dq, dk_, dv_ = (torch.empty_like(P[k]) for k in ("q", "k", "v"))
    dh0 = torch.empty_like(hT)
    img = gla.state_images(P["q"], P["v"])
    q, k, v, ld = P["q"], P["k"], P["v"], P["log_decay"]

    def plain():
        gla.gla_chunk_fwd(q, k, v, ld, None, out, hT, w.chunk, None, stream)
        gla.gla_chunk_bwd(q, k, v, do, ld, None, None, dq, dk_, dv_, dh0, w.chunk, None, stream)

    def saved():
        gla.gla_chunk_fwd_save(q, k, v, ld, None, out, hT, img, w.chunk, None, stream)
        gla.gla_chunk_bwd_saved(q, k, v, do, ld, None, None, img, dq, dk_, dv_, dh0, w.chunk, None, stream)

    res = {}
    for name, fn in (("plain_ms", plain), ("saved_states_ms", saved)):
        for _ in range(3):
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.bwd_steps)]
        for e in ev:
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    st_code = gla.gla_last_device_status(stream)
    if st_code != 0:
        raise SystemExit(f"device status after the training step: {st_code} ({gla.gla_status_str(st_code)})")
    res.update({"value": w.B * w.T / (res["saved_states_ms"] / 1e3), "unit": "tokens/s",
                "state_image_bytes": img.numel() * 2, "steps": args.bwd_steps,
                "note": "forward + backward of the layer; saved_states: the forward writes the state before every "
                        "chunk and the backward skips its forward state pass"})
    return res


def run_e2e(args, P, D, w, wd, out, hT, dout, stream):
    """Same step through the public API with host buffers.  Prefill: gla_chunk_fwd_host on pinned host
    q, k, v, log_decay (and h0 when the workload has one), writing out and hT to pinned host memory;
    the entry point overlaps copy-in, compute and copy-out by groups of sequences.  Decode: pinned
    q, k, v copied in, gla_decode_step, the output copied back; the state stays on the device."""
    import torch
    from gated_linear_rnn_gb300 import gla
    host = {k: P[k].cpu().pin_memory() for k in ("q", "k", "v", "log_decay")}
    h_h0 = None if P["h0"] is None else P["h0"].cpu().pin_memory()
    hostd = {k: D[k].cpu().pin_memory() for k in ("q", "k", "v")}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_hT = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
    h_dout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
    eq, ek, evv = (torch.empty_like(D[k]) for k in ("q", "k", "v"))
    nbytes = lambda ts: sum(t.numel() * t.element_size() for t in ts if t is not None)  # noqa: E731
    h2d_pre = nbytes(list(host.values()) + [h_h0])
    d2h_pre = nbytes((h_out, h_hT))
    h2d = h2d_pre + nbytes(hostd.values())
    d2h = d2h_pre + nbytes((h_dout,))
    steps = max(1, min(args.steps, 10))

    def prefill_step():
        gla.gla_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_decay"], h_h0, h_out, h_hT, w.chunk,
                               stream)

    def decode_step():
        eq.copy_(hostd["q"], non_blocking=True)
        ek.copy_(hostd["k"], non_blocking=True)
        evv.copy_(hostd["v"], non_blocking=True)
        gla.gla_decode_step(eq, ek, evv, D["log_decay"], D["state"], dout, stream)
        h_dout.copy_(dout, non_blocking=True)

    for _ in range(2):
        prefill_step()
        decode_step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        evs[i][0].record(stream)
        prefill_step()
        evs[i][1].record(stream)
        decode_step()
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    sbytes, _ = decode_bytes(wd.B, wd.H, wd.dk, wd.dv)
    return {"value": w.B * w.T / (pre_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "prefill_ms": pre_ms, "decode_ms": dec_ms, "steps": steps,
            "prefill_copy_gbs": (h2d_pre + d2h_pre) / (pre_ms / 1e3) / 1e9,
            "decode_state_gbs": sbytes / (dec_ms / 1e3) / 1e9,
            "note": "prefill through gla_chunk_fwd_host (pinned host arrays in and out, copies overlapped "
                    "with compute by groups of sequences); decode: pinned q,k,v in, out back, state resident"}


def run_only(args):
    """W + K back-to-back calls of one operation (the backward of the layer workload, the conv over
    B8 T2048 D3072, the forward of a prefill workload, or the gated forward of the layer workload), then a
    device-status check: a fixed command line to put under a profiler."""
    import torch
    from gated_linear_rnn_gb300 import build as Bld
    from gated_linear_rnn_gb300 import gla
    from gated_linear_rnn_gb300 import inputs as I
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    Bld.build_library()
    gla.load()
    w = I.WORKLOADS["layer_bf16"]
    if args.only in ("layer", "long", "ragged", "gated"):
        wp = I.WORKLOADS["layer_bf16" if args.only in ("layer", "gated") else "long_bf16" if args.only == "long"
                         else "ragged"]
        d = I.make_prefill(wp, device=dev, seed=0)
        cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].to(dev)
        nseq = d["q"].shape[0] if cu is None else cu.numel() - 1
        out = torch.empty(d["q"].shape[:3] + (wp.dv,), dtype=torch.bfloat16, device=dev)
        hT = torch.empty(nseq, wp.H, wp.dk, wp.dv, dtype=torch.float32, device=dev)

        g = I.make_gate(out.shape, device=dev, seed=5) if args.only == "gated" else None

        def call():
            if g is None:
                gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, wp.chunk, cu)
            else:
                gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["log_decay"], d["h0"], out, hT, wp.chunk, None,
                                        gate_kind=gla.GATE_SILU)
    elif args.only == "backward":
        d = I.make_backward(w, device=dev, seed=0, dhT_std=0.0)
        dq, dk, dv = (torch.empty_like(d[k]) for k in ("q", "k", "v"))

        def call():
            gla.gla_chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], None, None, dq, dk, dv, None, w.chunk)
    else:
        g = torch.Generator(device=dev).manual_seed(11)
        x = torch.randn(w.B, w.T, 3072, generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty_like(x)
        wt = torch.randn(3072, 4, generator=g, device=dev) * 0.5
        bias = torch.randn(3072, generator=g, device=dev) * 0.1

        def call():
            gla.gla_conv1d_silu(x, wt, bias, None, None, y)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    st_code = gla.gla_last_device_status()
    print(json.dumps({"only": args.only, "calls": args.warmup + args.steps, "status": st_code}), flush=True)
    return 0 if st_code == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-steps", type=int, default=5, help="timed launches of the backward (0: skip)")
    ap.add_argument("--only", choices=["backward", "conv", "layer", "long", "ragged", "gated"], default=None,
                    help="run just W + K calls of one operation on its bench workload (for profilers): the "
                         "layer backward, the conv, the forward of the layer, long-context or ragged "
                         "workload, or the gated forward of the layer workload (SiLU gate); prints one status "
                         "line, not the bench line")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of fp64 reference work to time")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only is not None:
        return run_only(args)
    if args.impl == "reference":
        # the CPU reference arm: rank 0 alone works, no process group is needed
        world, rank, _ = dist_setup(init=False)
        return run_reference(args, world, rank)
    world, rank, local = dist_setup()
    try:
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
