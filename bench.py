#!/usr/bin/env python
"""Benchmark of the KDA layer on GB300: prefill tokens/s and decode steps/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload layer_8k|varlen_16|long_1m] [--decode-steps K2]

Prefill step: one kda_prefill call over the whole batch (every stage of the
layer: conv + SiLU + L2, chunkwise gated delta rule, RMSNorm + gate, final
states).  Decode step: one kda_decode_step over 256 sequences x 96 heads.
Inputs are seeded synthetic data resident in HBM before the timed region;
every prefill batch (>= 1.2 GB of inputs) and the decode state (1.6 GB) are
larger than the 129 MB L2, so no flush is needed between iterations.

One JSON line is printed by rank 0.  With N > 1 ranks (torchrun), every rank
runs its own replica of the workload on its own GPU (units are independent:
no collective on the data path); the timed region is bracketed by barriers
and the slowest rank's time is used; value = all ranks' tokens / that time.

``--impl reference`` times the fp64 CPU oracle (the reference for this
layer) on the host cores, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=96,d=128) + decode steps/s; % of tensor/HBM roofline"
PREFILL_FLOP_PER_TOKEN_HEAD = {(128, 64): 180_224}   # 2C(3dk+2dv) + 6 dk dv
PREFILL_BYTES_PER_TOKEN_HEAD_BF16 = 1796             # q,k,v 768 + gate 256 + g 512 + beta 4 + y 256
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def aggregate_rate(world: int, units_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank; the slowest rank took ms_max."""
    return world * units_per_rank / (ms_max / 1e3)


def max_over_ranks(pg, x: float, device) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- helpers

def kernel_source_hash(files):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kimi_delta_attention_16_gb300", "csrc")
    for name in files:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str):
    """Per-launch DRAM bytes from a committed ncu summary, if the kernels have not changed."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel_key)
    except (ValueError, OSError):
        return None
    if not d or d.get("source_hash") != kernel_source_hash(d.get("files", [])):
        return None
    return d.get("bytes_per_launch")


def prefill_path(inp):
    """(path, segments, workspace bytes) of the kda_prefill calls on this batch."""
    from kimi_delta_attention_16_gb300 import kda_prefill_plan, kda_prefill_workspace_size
    path, segments = kda_prefill_plan(inp.T, inp.H, inp.D, N=inp.N, chunk=inp.chunk)
    ws = kda_prefill_workspace_size(inp.T, inp.H, inp.D, N=inp.N, chunk=inp.chunk)
    return path, segments, ws


def prefill_launches(path, segments):
    # kernels one kda_prefill call enqueues here (host cu_seqlens given, no conv_state_out):
    # tensor-core path: the fused chunk kernel, plus the segment composition and the output
    # fix-up when sequences are cut into segments; SIMT path: conv, chunk recurrence, epilogue.
    if path == "tc":
        return 1 if segments == 1 else 3
    return 3


# ----------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth

    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    if args.mode == "decode":
        return run_decode_only(args, world, rank, local, pg, dev, peaks, peak_src)
    if args.mode == "verify":  # profiling aid: only the multi-token decode loop
        obj, _ = time_multi_token(args, pg, dev, torch.cuda.current_stream(), peaks, peak_src, world)
        if rank == 0:
            print(f"multi-token decode {obj['metric']}: {obj['ms_per_step']:.4f} ms/step, "
                  f"{obj['roofline']['frac']:.3f} of HBM", flush=True)
        return
    if args.mode == "backward":  # profiling aid: only the backward pass (prints its object)
        obj, _ = time_backward(args, pg, dev, torch.cuda.current_stream(), peaks, peak_src, world)
        if rank == 0:
            print(json.dumps(obj))
        return
    if args.mode == "gemm":  # profiling aid: only the projection GEMMs of the projected layer
        return run_gemm_only(args, rank, dev)
    if args.mode == "prefill":
        args.decode_steps = 0
        args.verify_steps = 0
    if args.tokens:  # a shorter case of the same workload (profiling captures)
        inp = synth.make_prefill(args.workload, seed=1, device=dev, T=args.tokens,
                                 N=synth.WORKLOADS[args.workload]["N"])
    else:
        inp = synth.make_prefill(args.workload, seed=1, device=dev)
    N, T, H, D = inp.N, inp.T, inp.H, inp.D
    path, segments, ws_bytes = prefill_path(inp)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, D, D), dtype=torch.float32, device=dev)
    cu_dev = (torch.from_numpy(inp.cu_seqlens).to(dev), inp.cu_seqlens)  # (device, host)

    def step():
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, cu_dev, chunk=inp.chunk,
                        gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                        final_state=fin, out=out, workspace=ws)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(pg, ms, dev)
    tokens_per_s = aggregate_rate(world, T, ms_max)

    # roofline of the prefill launch(es)
    roof = prefill_roofline(inp, ms, path, segments, peaks, peak_src, args.workload)

    # end to end: every step copies its inputs from pinned host memory, runs kda_prefill and
    # reads its output and final state back.  The host link carries ~1.4 GB per step at about
    # 190 GB/s (both directions share it), so the copies run on their own streams with double
    # buffers: step i+1's inputs arrive while step i computes, and step i's results leave
    # behind it.  Every byte of every step still crosses the link inside the timed region.
    host = {}
    for name in ("q", "k", "v", "gate", "g", "beta"):
        t = getattr(inp, name)
        host[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[name].copy_(t)
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    fin_h = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
    dev_in = [{k: torch.empty_like(getattr(inp, k)) for k in host} for _ in range(2)]
    outs, fins = [out, torch.empty_like(out)], [fin, torch.empty_like(fin)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b have landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step using buffer b has computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of buffer b have been read back

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[b])
            for k in host:
                dev_in[b][k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])
        x = dev_in[b]
        kda.kda_prefill(x["q"], x["k"], x["v"], inp.conv_w, x["g"], x["beta"], cu_dev,
                        chunk=inp.chunk, gate=x["gate"], rms_w=inp.rms_w,
                        initial_state=inp.initial_state, final_state=fins[b], out=outs[b],
                        workspace=ws)
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            out_h.copy_(outs[b], non_blocking=True)
            fin_h.copy_(fins[b], non_blocking=True)
            ev_out[b].record(s_out)

    def e2e_run(n):
        start = torch.cuda.Event()
        start.record(stream)
        for e in ev_done + ev_out:
            e.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            e2e_step(i)
        stream.wait_event(ev_out[(n - 1) % 2])
        stream.wait_event(ev_out[n % 2])

    e2e_steps = max(2, min(args.steps, 10))
    e2e_run(2)
    torch.cuda.synchronize()
    barrier(pg)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1) / e2e_steps, dev)
    del host, dev_in, out_h, fin_h, outs, fins

    # decode: 256 sequences x 96 heads, one launch per step
    dec_obj = None
    dec_launches = 0
    if args.decode_steps > 0:
        del ws
        dec = synth.make_decode(seed=4, device=dev, N=args.decode_n)
        dout = torch.empty((dec.N, dec.H, dec.D), dtype=torch.bfloat16, device=dev)

        def dstep(i):
            j = i % dec.ring
            kda.kda_decode_step(dec.q[j], dec.k[j], dec.v[j], dec.g[j], dec.beta[j], dec.conv_w,
                                dec.state, dec.conv_state, gate=dec.gate[j], rms_w=dec.rms_w,
                                out=dout)

        for i in range(max(args.warmup, 3)):
            dstep(i)
        torch.cuda.synchronize()
        barrier(pg)
        e0.record(stream)
        for i in range(args.decode_steps):
            dstep(i)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(pg)
        dms = e0.elapsed_time(e1) / args.decode_steps
        dms_max = max_over_ranks(pg, dms, dev)
        Nd, Hd, Dd = dec.N, dec.H, dec.D
        dbytes = (2 * Nd * Hd * Dd * Dd * 4 + 2 * Nd * 3 * Hd * Dd * 3 * 2 + 4 * Nd * Hd * Dd * 2 +
                  Nd * Hd * Dd * 4 + Nd * Hd * 4 + Nd * Hd * Dd * 2)
        dgbs = dbytes / (dms / 1e3) / 1e9
        dec_launches = args.decode_steps
        dec_obj = {"metric": "KDA decode steps/s (256 seqs x 1 token, H=96, d=128)",
                   "value": round(world / (dms_max / 1e3), 2), "unit": "steps/s",
                   "tokens_per_s": round(world * Nd / (dms_max / 1e3), 1),
                   "ms_per_step": round(dms_max, 4), "steps": args.decode_steps,
                   "roofline": {"kernel": "k_decode", "bound": "hbm", "achieved": round(dgbs, 1),
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": round(dgbs / peaks["hbm_gbs"], 4),
                                "peak_source": peak_src,
                                "traffic": recorded_traffic("decode_decode_256"),
                                "algorithmic_bytes": dbytes}}
    # multi-token decode (speculative verification): 256 sequences x 4 new tokens per step
    mt_obj = None
    mt_launches = 0
    if args.verify_steps > 0:
        mt_obj, mt_launches = time_multi_token(args, pg, dev, stream, peaks, peak_src, world)
    # the other two prefill workloads, each its own nested key
    extra, extra_launches = {}, 0
    if args.extra_workloads and args.mode == "all" and not args.tokens:
        for name in ("varlen_16", "long_1m"):
            if name == args.workload:
                continue
            extra[name], nl = time_prefill_workload(name, args, pg, dev, stream, peaks, peak_src, world)
            extra_launches += nl
        extra["projected_layer"], nl = time_projected_layer(args, pg, dev, stream, peaks, peak_src, world)
        extra_launches += nl
        extra["backward"], nl = time_backward(args, pg, dev, stream, peaks, peak_src, world)
        extra_launches += nl
    clk = clocks.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, args.workload)

    if rank == 0:
        line = {"metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if path == "tc" else "fp32",
                "data": "synthetic",
                "config": {"workload": workload_desc(args.workload) +
                           (f" (shortened to T={T} for a profile)" if args.tokens else ""),
                           "global_batch": N * world,
                           "seq_len": T, "heads": H, "head_dim": D, "chunk": inp.chunk,
                           "prefill_path": path, "segments": segments, "l2": "inputs larger than L2 (no flush)",
                           "parallelism": f"replicas x{world}"},
                "roofline": roof,
                "e2e": {"value": round(world * T / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": round(e2e_ms, 4),
                        "note": "pinned host buffers; copies on their own streams, double-"
                                "buffered and overlapped with the neighbouring steps' compute"},
                "decode": dec_obj, "multi_token_decode": mt_obj, **extra, "cpu_baseline": cpu,
                "clocks": clk,
                "gpu_launches": (prefill_launches(path, segments) * args.steps + dec_launches + mt_launches +
                                 extra_launches)}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def prefill_roofline(inp, ms, path, segments, peaks, peak_src, workload):
    """Roofline object of one kda_prefill call: algorithmic bytes (and FLOPs) / CUDA-event time."""
    T, H, D, N = inp.T, inp.H, inp.D, inp.N
    fl = PREFILL_FLOP_PER_TOKEN_HEAD.get((D, inp.chunk), 0) * T * H
    state_bytes = N * H * D * D * 4 * (2 if inp.initial_state is not None else 1)
    alg_bytes = T * H * PREFILL_BYTES_PER_TOKEN_HEAD_BF16 + state_bytes
    gbs = alg_bytes / (ms / 1e3) / 1e9
    tflops = fl / (ms / 1e3) / 1e12
    kname = ("fused tcgen05 chunk kernel" if segments == 1 else
             f"fused tcgen05 chunk kernel, {segments} segments per sequence + composition + fix-up"
             ) if path == "tc" else "SIMT path: conv + chunk recurrence + epilogue"
    return {"kernel": "kda_prefill (" + kname + ")",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_src,
            "traffic": recorded_traffic(f"prefill_{path}_{workload}"),
            "algorithmic_bytes": alg_bytes, "algorithmic_flops": fl,
            "tensor_tflops": round(tflops, 1),
            "tensor_frac": round(tflops / peaks["bf16_tflops"], 4)}


def time_prefill_workload(name, args, pg, dev, stream, peaks, peak_src, world):
    """One more prefill workload (varlen_16 or long_1m), inputs resident in HBM, timed like the
    headline: warm-up calls, then K calls between CUDA events; returns (object, launches)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    inp = synth.make_prefill(name, seed=2 if name == "varlen_16" else 3, device=dev)
    N, T, H, D = inp.N, inp.T, inp.H, inp.D
    path, segments, ws_bytes = prefill_path(inp)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, D, D), dtype=torch.float32, device=dev)
    cu_pair = (torch.from_numpy(inp.cu_seqlens).to(dev), inp.cu_seqlens)

    def step():
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, cu_pair, chunk=inp.chunk,
                        gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                        final_state=fin, out=out, workspace=ws)

    steps = max(3, min(args.steps, 10))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / steps, dev)
    obj = {"metric": f"KDA prefill tokens/s ({name})", "value": round(aggregate_rate(world, T, ms), 1),
           "unit": "tokens/s", "ms_per_step": round(ms, 4), "steps": steps,
           "config": {"workload": workload_desc(name), "sequences": N, "tokens": T, "heads": H,
                      "head_dim": D, "chunk": inp.chunk, "prefill_path": path, "segments": segments},
           "roofline": prefill_roofline(inp, ms, path, segments, peaks, peak_src, name)}
    del inp, ws, out, fin
    torch.cuda.empty_cache()
    return obj, prefill_launches(path, segments) * steps


def time_projected_layer(args, pg, dev, stream, peaks, peak_src, world, d_model=7168):
    """The layer_8k prefill with the projections around it on the tensor cores: x -> g
    (-5 sigmoid), beta (sigmoid), gate pre-activations -> kda_prefill -> y -> y W_o.  Weights
    are random (N(0, 1/fan_in), bf16), x ~ N(0, 1); q, k, v stay the synthetic raw projections.
    Returns (object, launches)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    inp = synth.make_prefill("layer_8k", seed=1, device=dev)
    T, H, D = inp.T, inp.H, inp.D
    HD = H * D
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)

    def rnd(n, k, std):
        return (torch.randn(n, k, generator=gen, device=dev) * std).to(torch.bfloat16)

    x = rnd(T, d_model, 1.0)
    wa, wb, wg = rnd(HD, d_model, d_model ** -0.5), rnd(H, d_model, d_model ** -0.5), rnd(HD, d_model, d_model ** -0.5)
    wo = rnd(d_model, HD, HD ** -0.5)
    g = torch.empty((T, HD), dtype=torch.float32, device=dev)
    beta = torch.empty((T, H), dtype=torch.float32, device=dev)
    gate = torch.empty((T, HD), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, d_model), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    cu_pair = (torch.from_numpy(inp.cu_seqlens).to(dev), inp.cu_seqlens)
    path, segments, ws_bytes = prefill_path(inp)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    gemms = {
        "alpha (x W_a^T, -5 sigmoid)": lambda: kda.kda_gemm(x, wa, epilogue="decay", out=g),
        "beta (x W_b^T, sigmoid)": lambda: kda.kda_gemm(x, wb, epilogue="sigmoid", out=beta),
        "gate (x W_g^T)": lambda: kda.kda_gemm(x, wg, epilogue="none", out=gate),
        "output (y W_o^T)": lambda: kda.kda_gemm(y.view(T, HD), wo, epilogue="none", out=out),
    }
    flops = {"alpha (x W_a^T, -5 sigmoid)": 2 * T * HD * d_model, "beta (x W_b^T, sigmoid)": 2 * T * H * d_model,
             "gate (x W_g^T)": 2 * T * HD * d_model, "output (y W_o^T)": 2 * T * d_model * HD}

    def step():
        for name in ("alpha (x W_a^T, -5 sigmoid)", "beta (x W_b^T, sigmoid)", "gate (x W_g^T)"):
            gemms[name]()
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, g.view(T, H, D), beta, cu_pair, chunk=inp.chunk,
                        gate=gate.view(T, H, D), rms_w=inp.rms_w, final_state=fin, out=y, workspace=ws)
        gemms["output (y W_o^T)"]()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, n):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        barrier(pg)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(pg)
        return max_over_ranks(pg, e0.elapsed_time(e1) / n, dev)

    steps = max(3, min(args.steps, 10))
    traffic_key = {"alpha (x W_a^T, -5 sigmoid)": "gemm_alpha", "gate (x W_g^T)": "gemm_gate",
                   "output (y W_o^T)": "gemm_output"}
    per = {}
    for name, fn in gemms.items():
        ms = timed(fn, steps)
        tf = flops[name] / (ms / 1e3) / 1e12
        per[name] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": recorded_traffic(traffic_key[name]) if name in traffic_key else None}
    ms = timed(step, steps)
    gemm_ms = sum(v["ms"] for v in per.values())
    gemm_flops = sum(flops.values())
    gemm_tf = gemm_flops / (gemm_ms / 1e3) / 1e12
    obj = {"metric": "KDA layer with its projections, tokens/s (layer_8k, d_model 7168)",
           "value": round(aggregate_rate(world, T, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "steps": steps,
           "config": {"workload": "layer_8k with x [8192, 7168] bf16 ~ N(0,1) and random bf16 weights "
                                  "N(0, 1/fan_in): W_a, W_g [12288, 7168], W_b [96, 7168], W_o [7168, 12288]; "
                                  "q, k, v synthetic raw projections", "prefill_path": path, "segments": segments},
           "gemms": per,
           "roofline": {"kernel": "k_gemm (tcgen05, 128x256 tiles, 4-stage TMA ring), the four projections",
                        "bound": "tensor", "achieved": round(gemm_tf, 1), "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": round(gemm_tf / peaks["bf16_tflops"], 4), "peak_source": peak_src,
                        "traffic": None, "algorithmic_flops": gemm_flops}}
    del x, wa, wb, wg, wo, g, beta, gate, y, out, ws, inp
    torch.cuda.empty_cache()
    # inside the timed regions: each projection alone, then the whole chain
    launches = len(gemms) * steps + (len(gemms) + prefill_launches(path, segments)) * steps
    return obj, launches


FP32_SIMT_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # 152 SMs x 128 fp32 lanes x FMA x 2.07 GHz max clock
TF32_PER_BF16 = 1.1 / 2.25                            # nominal dense TF32 / bf16 tensor rates
BWD_FLOP_PER_TOKEN_HEAD = 28 * 128 * 128              # four token-serial sweeps of the state, 7 d^2 each


def time_backward(args, pg, dev, stream, peaks, peak_src, world):
    """kda_backward at layer_8k (8192 tokens, 96 heads): the gradients of every input given dy and
    dS_fin, with the gate, RMSNorm weight, initial state and conv state present.  Workspace and
    outputs are allocated once, outside the timed region.  Returns (object, launches)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    short = {"T": args.tokens} if args.tokens else {}  # a shorter case of the same workload (profiles)
    inp = synth.make_prefill("layer_8k", seed=1, device=dev, s0_std=0.02, conv_state=True, rms_w="random",
                             **short)
    T, H, D, N = inp.T, inp.H, inp.D, inp.N
    gen = torch.Generator(device=dev)
    gen.manual_seed(9)
    dy = torch.randn((T, H, D), generator=gen, device=dev).to(torch.bfloat16)
    dsf = torch.randn((N, H, D, D), generator=gen, device=dev) * 0.02
    cu_pair = (torch.from_numpy(inp.cu_seqlens).to(dev), inp.cu_seqlens)
    ws = torch.empty(kda.kda_backward_workspace_size(inp.cu_seqlens, H), dtype=torch.uint8, device=dev)

    def step():
        kda.kda_backward(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, cu_pair, dy, gate=inp.gate,
                         rms_w=inp.rms_w, initial_state=inp.initial_state, conv_state_in=inp.conv_state_in,
                         d_final_state=dsf, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier(pg)
    steps = max(3, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / steps, dev)
    flops = BWD_FLOP_PER_TOKEN_HEAD * T * H
    tf = flops / (ms / 1e3) / 1e12
    # the recurrence products run on the tensor cores as TF32 (three hi/lo terms each): the peak of
    # that dtype is the measured bf16 peak times the nominal dense TF32 / bf16 ratio (1.1 / 2.25)
    tf32_peak = peaks["bf16_tflops"] * TF32_PER_BF16
    obj = {"metric": f"KDA backward tokens/s (layer_8k: T={T}, H=96, d=128; all input gradients)",
           "value": round(aggregate_rate(world, T, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "steps": steps, "workspace_bytes": ws.numel(),
           "roofline": {"kernel": "the whole kda_backward call (TF32 tcgen05 row sweeps and mma.sync chunk "
                                  "sweeps dominate, 3 hi/lo terms per product)",
                        "bound": "tensor", "achieved": round(tf, 2), "peak": round(tf32_peak, 1),
                        "unit": "TFLOP/s", "frac": round(tf / tf32_peak, 4),
                        "peak_source": f"{peak_src} bf16 x 1.1/2.25 (nominal dense TF32 / bf16)",
                        "fp32_simt_frac": round(tf / FP32_SIMT_TFLOPS, 4),
                        "traffic": None, "algorithmic_flops": flops}}
    del inp, dy, dsf, ws
    torch.cuda.empty_cache()
    return obj, steps * 10  # ten kernels per call (the five output/partial memsets are not counted)


def time_multi_token(args, pg, dev, stream, peaks, peak_src, world, t_new=4, ring=8):
    """kda_prefill on 256 sequences x t_new tokens continuing from carried states and conv
    states (the recurrent path): the decode workload's inputs, t_new consecutive tokens per
    call, from a ring of `ring` packed steps (larger than L2 together with the states)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    dec = synth.make_decode(seed=6, device=dev, N=args.decode_n, ring=t_new * ring)
    N, H, D = dec.N, dec.H, dec.D

    def pack(x, r):  # ring entries r*t_new .. +t_new-1 -> sequence-major token rows
        y = x[r * t_new:(r + 1) * t_new]
        return y.transpose(0, 1).reshape(N * t_new, *y.shape[2:]).contiguous()

    steps_in = [{k: pack(getattr(dec, k), r) for k in ("q", "k", "v", "gate", "g", "beta")}
                for r in range(ring)]
    cu = synth.cu_from_lengths([t_new] * N)
    cu_pair = (torch.from_numpy(cu).to(dev), cu)
    path = kda.kda_prefill_plan(N * t_new, H, D, cu_seqlens=cu)[0]
    out = torch.empty((N * t_new, H, D), dtype=torch.bfloat16, device=dev)
    cs = [dec.conv_state, torch.empty_like(dec.conv_state)]

    def mstep(i):
        x = steps_in[i % ring]
        kda.kda_prefill(x["q"], x["k"], x["v"], dec.conv_w, x["g"], x["beta"], cu_pair,
                        gate=x["gate"], rms_w=dec.rms_w, initial_state=dec.state,
                        final_state=dec.state, conv_state_in=cs[i % 2],
                        conv_state_out=cs[(i + 1) % 2], out=out)

    for i in range(max(args.warmup, 3)):
        mstep(i)
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.verify_steps):
        mstep(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.verify_steps, dev)
    T = N * t_new
    nbytes = (2 * N * H * D * D * 4 + 2 * N * 3 * H * D * 3 * 2 + 4 * T * H * D * 2 +
              T * H * D * 4 + T * H * 4 + T * H * D * 2)
    gbs = nbytes / (ms / 1e3) / 1e9
    obj = {"metric": f"KDA multi-token decode steps/s ({N} seqs x {t_new} tokens, H={H}, d={D})",
           "value": round(world / (ms / 1e3), 2), "unit": "steps/s",
           "tokens_per_s": round(world * T / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
           "steps": args.verify_steps, "prefill_path": path,
           "roofline": {"kernel": "k_short_tma (recurrent path; rolls the conv state itself)",
                        "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                        "peak_source": peak_src, "traffic": recorded_traffic("short_verify_256x4"),
                        "algorithmic_bytes": nbytes}}
    del steps_in, dec
    return obj, args.verify_steps  # one launch per call: the recurrent kernel also rolls the conv state


def run_gemm_only(args, rank, dev, d_model=7168, HD=12288):
    """Profiling aid: the alpha (-5 sigmoid), gate and output projections of the projected layer
    at T = --tokens (default 8192) tokens; prints each one's time (no JSON line)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    T = args.tokens or 8192
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)

    def rnd(n, k, std):
        return (torch.randn(n, k, generator=gen, device=dev) * std).to(torch.bfloat16)

    x, y = rnd(T, d_model, 1.0), rnd(T, HD, 1.0)
    wa, wg, wo = rnd(HD, d_model, d_model ** -0.5), rnd(HD, d_model, d_model ** -0.5), rnd(d_model, HD, HD ** -0.5)
    g = torch.empty((T, HD), dtype=torch.float32, device=dev)
    gate = torch.empty((T, HD), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, d_model), dtype=torch.bfloat16, device=dev)
    runs = {"alpha": lambda: kda.kda_gemm(x, wa, epilogue="decay", out=g),
            "gate": lambda: kda.kda_gemm(x, wg, epilogue="none", out=gate),
            "output": lambda: kda.kda_gemm(y, wo, epilogue="none", out=out)}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, fn in runs.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        if rank == 0:
            print(f"gemm {name} (T={T}): {ms:.4f} ms, {2 * T * HD * d_model / (ms / 1e3) / 1e12:.1f} TFLOP/s")


def run_decode_only(args, world, rank, local, pg, dev, peaks, peak_src):
    """Profiling aid: only the decode loop (no JSON line; prints the step time)."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    dec = synth.make_decode(seed=4, device=dev, N=args.decode_n)
    dout = torch.empty((dec.N, dec.H, dec.D), dtype=torch.bfloat16, device=dev)
    n = max(args.warmup, 3) + args.decode_steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(n):
        if i == n - args.decode_steps:
            e0.record()
        j = i % dec.ring
        kda.kda_decode_step(dec.q[j], dec.k[j], dec.v[j], dec.g[j], dec.beta[j], dec.conv_w,
                            dec.state, dec.conv_state, gate=dec.gate[j], rms_w=dec.rms_w, out=dout)
    e1.record()
    torch.cuda.synchronize()
    if rank == 0:
        print(f"decode N={dec.N}: {e0.elapsed_time(e1) / max(args.decode_steps, 1):.4f} ms/step")


def workload_desc(name):
    return {
        "layer_8k": "layer_8k: one KDA layer prefill, B=1, T=8192, H=96, d=128, chunk 64, bf16 "
                    "q/k/v/gate, fp32 g/beta/state, zero initial state",
        "varlen_16": "varlen_16: 16 packed sequences, lengths log-uniform in [512,16384], H=96, "
                     "d=128, bf16 I/O, initial states N(0,0.02^2)",
        "long_1m": "long_1m: B=1, T=1048576, H=24, d=128, chunk 64, bf16 I/O",
    }[name]


# ----------------------------------------------------------------------------- oracle timing

def cpu_baseline(inp, workload, tokens=None):
    """The fp64 oracle, as it stands, on a bounded sample of the same workload."""
    import oracle
    from kimi_delta_attention_16_gb300 import synth
    import numpy as np
    # the first sequence, capped at 8192 tokens (about 1e11 fp64 flop at H=96, d=128)
    n_tok = tokens or min(int(inp.cu_seqlens[1]), 8192)
    s = slice(0, n_tok)
    f = synth.to_f32_numpy
    a = dict(q=f(inp.q[s]), k=f(inp.k[s]), v=f(inp.v[s]), conv_w=f(inp.conv_w),
             cu_seqlens=np.array([0, n_tok], np.int32), g=f(inp.g[s]), beta=f(inp.beta[s]),
             gate=f(inp.gate[s]) if inp.gate is not None else None, rms_w=f(inp.rms_w),
             initial_state=None if inp.initial_state is None else f(inp.initial_state[:1]))
    cores = min(oracle.num_cores(), inp.H)
    t0 = time.perf_counter()
    oracle.forward(**a, n_threads=cores)
    dt = time.perf_counter() - t0
    return {"value": round(n_tok / dt, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n_tok} tokens of the first sequence, all {inp.H} heads "
                      f"({workload}), fp64 token-sequential oracle, {dt:.2f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch  # noqa: F401  (CPU tensors only)
    from kimi_delta_attention_16_gb300 import synth
    import oracle
    w = synth.WORKLOADS[args.workload]
    sample_tokens = 256
    inp = synth.make_prefill(args.workload, seed=1, device="cpu",
                             lengths=[sample_tokens], H=w["H"], D=w["D"])
    times = []
    res = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        res = cpu_baseline(inp, args.workload, tokens=sample_tokens)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = statistics.mean(times) if times else float("nan")
    value = sample_tokens / per_step
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "seq_len": w.get("T"),
                       "heads": w["H"], "head_dim": w["D"]},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": res["cores"],
                             "kind": "oracle",
                             "sample": f"each step: {sample_tokens} tokens x {w['H']} heads of "
                                       f"{args.workload} through the fp64 oracle"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["layer_8k", "varlen_16", "long_1m"], default="layer_8k")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--decode-n", type=int, default=256, help="decode batch (sequences)")
    ap.add_argument("--verify-steps", type=int, default=200,
                    help="multi-token decode steps (256 sequences x 4 tokens) to time; 0 skips")
    ap.add_argument("--mode", choices=["all", "prefill", "decode", "verify", "gemm", "backward"], default="all",
                    help="profiling aid: run only one of the measurements (verify = the "
                         "multi-token decode loop, gemm = the projection GEMMs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", dest="extra_workloads", action="store_false",
                    help="skip the nested varlen_16 and long_1m prefill measurements")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling aid: total tokens of a shorter case of --workload")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
