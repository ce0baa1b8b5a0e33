#!/usr/bin/env python3
"""Benchmark of the TP-MLP block forward+backward on one GB300 (t logical shards).

Workload (one "step"): the 2048-token TP MLP with h = 4096, F = 16384, t = 4,
GeLU(tanh), biases -- column-parallel GEMM + activation, row-parallel GEMM with
the fused g reduction, then the backward (dgrad with act', both wgrads, the f
reduction of dX, bias grads) -- on synthetic seeded bf16 inputs resident in
HBM.  FLOPs counted: the six GEMMs, 12 * M * h * F = 1.649e12 per step.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead (the only other arm: the pages publish no implementation).  Under
torchrun with N > 1 every rank runs an independent replica on its own GPU
(the t shards are logical and live on one GPU, so there is nothing to
exchange between GPUs); value = all ranks' work / max-over-ranks time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TP-MLP block fwd+bwd TFLOP/s on 1 GB300 (t logical shards), % of bf16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "c2"


def flops_per_step(M, h, F):
    return 12.0 * M * h * F


# --------------------------------------------------------------------- ranks

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def reduce_max(dist, value):
    """Max over ranks of one float (host-side, gloo)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate(units_per_rank, seconds_max, world):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling in the background; each line is stamped on arrival."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id=None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id:
            cmd[1:1] = ["-i", gpu_id]
        self.samples = []
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        window = [p for ts, p in self.samples if t0 - 0.15 <= ts <= t1 + 0.15]
        if not window:   # timed region shorter than the sampling period: nearest samples under load
            window = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1]]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in window if num(p[0]) is not None]
        mx = [num(p[1]) for p in window if num(p[1]) is not None]
        reasons = sorted({n for p in window for n, v in zip(self.NAMES, p[3:7]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(window)}


# -------------------------------------------------------------- peaks, traffic

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"bf16_burst": float(d["bf16_tflops"]), "bf16_sustained": float(d["bf16_tflops_sustained"]),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def gemm_source_hash():
    h = hashlib.sha256()
    for name in ("gemm.cu", "ptx.cuh", "devmath.cuh"):
        with open(os.path.join(ROOT, "megatron_tensor_transformer_shard_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip().lstrip("- ").strip("`")] = v.strip().strip("`")
        if kv.get("source_sha") != gemm_source_hash():
            return None
        return float(kv["dram_bytes_per_launch_full_size"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    rank, world, local = dist_env()
    dist = init_dist(world)
    torch.cuda.set_device(local)
    from megatron_tensor_transformer_shard_gb300 import build as B
    B.build()
    from megatron_tensor_transformer_shard_gb300 import _lib as L
    from megatron_tensor_transformer_shard_gb300 import inputs as I

    cfg = I.CONFIGS[WORKLOAD]
    M, h, F, t, act = cfg["M"], cfg["h"], cfg["F"], cfg["t"], L.ACT_BY_NAME[cfg["act"]]
    Ft = F // t
    dev = "cuda"
    # Seeded synthetic inputs drawn on the device (same distributions as the parity tests).
    inp = I.mlp_inputs(M, h, F, bias=True, dy=True, seed=rank, device=dev)
    bf16, f32 = torch.bfloat16, torch.float32
    Wup_p = torch.empty(t, Ft, h, dtype=bf16, device=dev)
    Wdown_p = torch.empty(t, h, Ft, dtype=bf16, device=dev)
    L.tp_pack_col(inp["W_up"], h, F, t, Wup_p)
    L.tp_pack_row(inp["W_down"], F, h, t, Wdown_p)
    X, dY, bup, bdown = inp["X"], inp["dY"], inp["b_up"], inp["b_down"]
    del inp["W_up"], inp["W_down"]
    Y = torch.empty(M, h, dtype=bf16, device=dev)
    Z = torch.empty(t, M, Ft, dtype=bf16, device=dev)
    A = torch.empty_like(Z)
    dX = torch.empty(M, h, dtype=bf16, device=dev)
    dWup = torch.empty(t, Ft, h, dtype=f32, device=dev)
    dWdown = torch.empty(t, h, Ft, dtype=f32, device=dev)
    dbup = torch.empty(F, dtype=f32, device=dev)
    dbdown = torch.empty(h, dtype=f32, device=dev)
    nws = L.tp_mlp_backward_workspace_size(M, h, F, t, 0)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    # forward GEMMs' workspace (split-K partials); the calls run one after the other
    nfw = max(L.tp_column_parallel_workspace_size(M, h, F, t), L.tp_row_parallel_workspace_size(M, F, h, t))
    fws = torch.empty(nfw, dtype=torch.uint8, device=dev)

    col_ev = []

    def run_step(X, dY, Y, dX, record=False):
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        # forward: f (identity) + column-parallel GEMM + GeLU, then row-parallel GEMM + g (bias once)
        L.tp_column_parallel_forward_ws(X, M, h, F, t, act, Wup_p, bup, Z, A, fws, nfw)
        if record:
            e1.record()
            col_ev.append((e0, e1))
        L.tp_row_parallel_forward_ws(A, M, F, h, t, Wdown_p, bdown, None, Y, fws, nfw)
        # backward: g (identity), dgrad*act', wgrads, f (fused dX reduction), bias grads
        L.tp_mlp_backward(dY, X, Z, A, M, h, F, t, act, Wup_p, Wdown_p, dX, dWup, dWdown, dbup, dbdown, 0, 0,
                          ws, nws)

    def step(record=False):
        run_step(X, dY, Y, dX, record)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if L.tp_get_device_status(check=False) != L.TP_OK:
        raise RuntimeError("device error during warm-up")

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)

    stream = torch.cuda.current_stream()
    barrier(dist)
    torch.cuda.synchronize()
    n0 = L.tp_kernel_launch_count()
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev_a.record(stream)
    for _ in range(args.steps):
        step(record=True)
    ev_b.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(dist)
    launches = L.tp_kernel_launch_count() - n0
    status = L.tp_get_device_status(check=False)
    if status != L.TP_OK:
        raise RuntimeError(f"device error in timed region: {L.status_string(status)}")
    ms = ev_a.elapsed_time(ev_b) / args.steps
    ms_max = reduce_max(dist, ms)
    col_ms = statistics.mean(a.elapsed_time(b) for a, b in col_ev)
    clk = clocks.summary(t_wall0, t_wall1) if clocks else None

    # end to end: host (pinned) inputs copied in, results read back, every step
    e2e = None
    if not args.no_e2e:
        Xh = torch.empty(M, h, dtype=bf16, pin_memory=True).copy_(X.cpu())
        dYh = torch.empty(M, h, dtype=bf16, pin_memory=True).copy_(dY.cpu())
        Yh = torch.empty(M, h, dtype=bf16, pin_memory=True)
        dXh = torch.empty(M, h, dtype=bf16, pin_memory=True)

        # As a training loop with a pinned-memory prefetcher runs it: two device buffer sets
        # and a copy stream, so step k+1's inputs go up and step k's results come down while
        # step k / k+1 computes.  Every copy is inside the timed region: the copy stream starts
        # after the start event and the end event follows the last download.
        Xd, dYd = [X, torch.empty_like(X)], [dY, torch.empty_like(dY)]
        Yd, dXd = [Y, torch.empty_like(Y)], [dX, torch.empty_like(dX)]
        copy = torch.cuda.Stream()
        up = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_run(nsteps, start_ev=None):
            with torch.cuda.stream(copy):
                if start_ev is not None:
                    copy.wait_event(start_ev)
                else:
                    copy.wait_stream(stream)
                Xd[0].copy_(Xh, non_blocking=True)
                dYd[0].copy_(dYh, non_blocking=True)
                up[0].record(copy)
            for k in range(nsteps):
                c, n = k % 2, 1 - k % 2
                stream.wait_event(up[c])
                run_step(Xd[c], dYd[c], Yd[c], dXd[c])
                done[c].record(stream)
                with torch.cuda.stream(copy):
                    if k + 1 < nsteps:
                        if k >= 1:
                            copy.wait_event(done[n])  # buffer n was step k-1's
                        Xd[n].copy_(Xh, non_blocking=True)
                        dYd[n].copy_(dYh, non_blocking=True)
                        up[n].record(copy)
                    copy.wait_event(done[c])
                    Yh.copy_(Yd[c], non_blocking=True)
                    dXh.copy_(dXd[c], non_blocking=True)
            stream.wait_stream(copy)

        e2e_run(max(1, args.warmup))
        barrier(dist)
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        e2e_run(args.steps, ea)
        eb.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        if not torch.equal(Yh, Yd[(args.steps - 1) % 2].cpu()):
            raise RuntimeError("end-to-end read-back does not match the device result")
        e_ms = reduce_max(dist, ea.elapsed_time(eb) / args.steps)
        e2e = {"value": round(aggregate(flops_per_step(M, h, F), e_ms / 1e3, world) / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": 2 * M * h * 2, "d2h_bytes_per_step": 2 * M * h * 2,
               "copies": "pinned host buffers; uploads and read-backs on a copy stream, overlapped with the "
                         "neighbouring steps' compute (double-buffered device inputs / outputs)"}

    if clocks:
        clocks.stop()

    secondary = None
    if not args.no_extras and rank == 0:
        del Z, A, dWup, dWdown, ws
        torch.cuda.empty_cache()
        full = {"layer_c4": run_layer_extra(L, torch, args, "c4"),
                "sp_layer_c5": run_layer_extra(L, torch, args, "c5"),
                "attention_c5": run_attn_extra(L, torch, args, "c5"),
                "sp_layernorm_c5": run_ln_extra(L, torch, args, "c5"),
                "decode_attention": run_decode_attn_extra(L, torch, args),
                "vocab_embedding": run_embedding_extra(L, torch, args),
                "row_parallel_overlap_c2": run_overlap_extra(L, torch, args),
                "mlp_fwd_c1": run_mlp_fwd_extra(L, torch, args),
                "decode_c3": run_decode_extra(L, torch, args)}
        # The full records (workload descriptions, byte counts) go to stderr; the JSON line
        # keeps a few numbers per workload, the two target workloads last.
        print(json.dumps({"secondary_detail": full}), file=sys.stderr, flush=True)
        secondary = {k: compact_secondary(k, v) for k, v in full.items()}

    if rank != 0:
        return None
    peaks = measured_peaks()
    region_s = ms * args.steps / 1e3
    peak_kind = "bf16_sustained" if region_s >= 2.0 else "bf16_burst"
    peak = peaks[peak_kind]
    col_flops = 2.0 * M * h * F
    achieved = col_flops / (col_ms / 1e3) / 1e12
    value = aggregate(flops_per_step(M, h, F), ms_max / 1e3, world) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "TP-MLP fwd+bwd, t=4, X 2048x4096, W_up 4096x16384, W_down 16384x4096, GeLU(tanh)",
                   "global_batch": M * world, "seq_len": M, "parallelism": f"t=4 logical shards x {world} replica(s)",
                   "l2": "working set ~1.1 GB > 129 MB L2; no flush",
                   "frac_of_peak": round(value / world / peak, 4), "peak_tflops": peak,
                   "peak_kind": f"{peak_kind} ({peaks['source']})"},
        "roofline": {"bound": "tensor", "kernel": "gemm_pair_kernel<K-major, K-major, EPI_ACT, GeLU-tanh> (column-parallel GEMM + GeLU epilogue; 512 tiles: whole rounds, no K split)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic("gemm_colpar_fwd_c2.md"),
                     "kernel_ms": round(col_ms, 4), "flops_per_launch": col_flops},
        "clocks": clk, "e2e": e2e, "gpu_launches": int(launches),
    }
    if world == 1 and not args.no_cpu_baseline:
        cb, parity = cpu_baseline(budget_s=args.cpu_budget, gpu=GpuMlp(L, torch), layers=args.cpu_layers)
        line["cpu_baseline"] = cb
        line["parity"] = parity
    if secondary:
        line["secondary"] = secondary
    return line


# Numbers kept in the JSON line per secondary workload (the rest goes to stderr).
_COMPACT = {
    "layer_c4": ("ms_per_step", "TFLOPs", "frac_of_peak"),
    "sp_layer_c5": ("ms_per_step", "TFLOPs", "frac_of_peak"),
    "attention_c5": ("fwd_ms", "bwd_ms", "core_fwd_ms", "core_fwd_TFLOPs", "core_bwd_ms", "core_bwd_TFLOPs"),
    "sp_layernorm_c5": ("fwd_us", "fwd_frac_of_hbm", "bwd_us", "bwd_frac_of_hbm"),
    "decode_attention": ("us_per_step", "frac_of_hbm", "us_per_step_graph"),
    "vocab_embedding": ("fwd_us", "fwd_frac_of_hbm", "bwd_us", "bwd_frac_of_hbm"),
    "row_parallel_overlap_c2": ("fused_ms", "fused_splitk_ms", "overlap_ms", "gemm_plus_reduce_ms"),
    "mlp_fwd_c1": ("us_per_step", "TFLOPs", "us_per_step_graph"),
    "decode_c3": ("us_per_step", "GBps", "frac_of_hbm", "frac_of_8TBps"),
}


def compact_secondary(name, rec):
    keys = _COMPACT.get(name)
    return {k: rec[k] for k in keys if k in rec} if keys else rec


class GpuMlp:
    """The TP-MLP path through the C ABI on host-drawn inputs (the parity leg of the
    oracle baseline compares its rows with the oracle's)."""

    def __init__(self, L, torch):
        self.L, self.torch = L, torch

    def run(self, inp_cpu, M, h, F, t, act_name, backward):
        L, torch = self.L, self.torch
        from megatron_tensor_transformer_shard_gb300 import tp as T
        d = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
        w = T.MLPWeights(d["W_up"], d["b_up"], d["W_down"], d["b_down"], t)
        Y, Z, A = T.mlp_forward(d["X"], w, act_name)
        out = {"Y": Y}
        if backward:
            out["dX"] = T.mlp_backward(d["dY"], d["X"], Z, A, w, act_name)["dX"]
        torch.cuda.synchronize()
        if L.tp_get_device_status(check=False) != L.TP_OK:
            raise RuntimeError("device error in the parity run")
        return {k: v.cpu() for k, v in out.items()}


def _time(torch, fn, iters, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters  # ms


def run_decode_extra(L, torch, args):
    """Decode-shaped SwiGLU GEMV (x 1x8192, W_gate/W_up 8192x28672, W_down
    28672x8192, t = 4): HBM GB/s of the whole decode step (two kernels)."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    c = I.CONFIGS["c3"]
    M, h, F, t = c["M"], c["h"], c["F"], c["t"]
    inp = I.swiglu_inputs(M, h, F, seed=0, device="cuda")
    Wgu = torch.empty(2 * F, h, dtype=torch.bfloat16, device="cuda")
    Wd = torch.empty(t, h, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_swiglu(inp["W_gate"], inp["W_up"], h, F, t, Wgu)
    L.tp_pack_row(inp["W_down"], F, h, t, Wd)
    del inp["W_gate"], inp["W_up"], inp["W_down"]
    y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    a = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    us = 1e3 * _time(torch, lambda: L.tp_decode_swiglu_forward(inp["X"], M, h, F, t, Wgu, Wd, y, a),
                     max(20, args.steps), warmup=5)
    nbytes = 3 * h * F * 2 + M * h * 2 * 2 + M * F * 2 * 2
    gbs = nbytes / (us / 1e6) / 1e9
    peaks = measured_peaks()
    return {"workload": "decode SwiGLU GEMV, t=4, x 1x8192, W_gate/W_up 8192x28672, W_down 28672x8192",
            "us_per_step": round(us, 2), "GBps": round(gbs, 1), "bytes_per_step": nbytes,
            "frac_of_hbm": round(gbs / peaks["hbm"], 4), "hbm_peak_GBps": peaks["hbm"],
            "frac_of_8TBps": round(gbs / 8000.0, 4), "l2": "1.41 GB of weights > L2; no flush"}


def run_decode_attn_extra(L, torch, args):
    """Decode attention over a head-sharded KV cache, Llama-3-70B-shaped at
    TP=4: d=8192, 64 query heads and 8 KV heads of 128 (two KV heads and their
    two 8-head groups per shard), 8 sequences whose cache lengths are drawn
    uniformly from 4096..8192 keys.  One step = QKV GEMV + cache append +
    split-KV attention + combine + W_o GEMV with the g sum."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    from megatron_tensor_transformer_shard_gb300 import tp as T
    nh, nkv, hd, t, B, L_max = 64, 8, 128, 4, 8, 8192
    d = nh * hd
    inp = I.decode_attn_inputs(B, d, nh, nkv, hd, L_max, bias=False, seed=0, device="cuda")
    pos = I.decode_positions(B, 4095, L_max - 1, seed=0)
    w = T.DecodeAttnWeights(inp["W_qkv"], None, inp["W_o"], None, nh, nkv, hd, t)
    del inp["W_qkv"], inp["W_o"]
    # n_kv = 8 >= t: shard i holds KV heads 2i, 2i+1, so the per-shard cache is the unsplit one
    K = inp["K"].view(w.cache_shape(B, L_max))
    V = inp["V"].view(w.cache_shape(B, L_max))
    posd = pos.cuda()
    ws = w.workspace(B, L_max, "cuda")
    x = inp["x"]
    y = torch.empty(B, d, dtype=torch.bfloat16, device="cuda")
    step = lambda: T.decode_attn_forward(x, w, K, V, posd, ws=ws, out=y)
    us = 1e3 * _time(torch, step, max(20, args.steps), warmup=5)
    # the same step replayed from a CUDA graph (how a decode loop launches it)
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        step()
        with torch.cuda.graph(graph, stream=cs):
            step()
    torch.cuda.current_stream().wait_stream(cs)
    us_graph = 1e3 * _time(torch, graph.replay, max(20, args.steps), warmup=5)
    R = (nh // t + 2 * w.kv_t) * hd
    w_bytes = t * R * d * 2 + nh * hd * d * 2
    kv_bytes = sum(2 * t * w.kv_t * (int(p) + 1) * hd * 2 for p in pos.tolist())
    nbytes = w_bytes + kv_bytes
    gbs = nbytes / (us / 1e6) / 1e9
    peaks = measured_peaks()
    return {"workload": "decode attention, t=4, d=8192, 64 query / 8 KV heads x 128, B=8, cache lengths "
                        "4096..8192 (seeded uniform), fp16 KV cache",
            "us_per_step": round(us, 2), "GBps": round(gbs, 1), "bytes_per_step": nbytes,
            "us_per_step_graph": round(us_graph, 2), "GBps_graph": round(nbytes / (us_graph / 1e6) / 1e9, 1),
            "weight_bytes": w_bytes, "kv_bytes": kv_bytes, "lengths": [int(p) + 1 for p in pos.tolist()],
            "frac_of_hbm": round(gbs / peaks["hbm"], 4), "hbm_peak_GBps": peaks["hbm"],
            "frac_of_hbm_graph": round(nbytes / (us_graph / 1e6) / 1e9 / peaks["hbm"], 4),
            "l2": "~500 MB of weights and cache per step > L2; no flush",
            "allreduce_accounting": {"payload_bytes": B * d * 2, "allreduces_per_layer_per_token": 2,
                                     "allreduces_per_token_80_layers": 160,
                                     "on_device": "each is the fixed-order shard sum inside the row-parallel "
                                                  "GEMV (W_o here, W_down in the MLP): no extra HBM bytes"}}


def run_embedding_extra(L, torch, args):
    """Vocab-parallel embedding, Llama-3-sized vocabulary: V = 128256, h = 8192,
    t = 4, 4096 Zipf-distributed token ids.  Forward = gather from the owning
    shard; backward accumulates into the shards' fp32 gradient rows."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    N, V, h, t = 4096, 128256, 8192, 4
    ids = I.token_ids(N, V, seed=0).cuda()
    inp = I.embedding_inputs(N, V, h, seed=0, device="cuda")
    Y = torch.empty(N, h, dtype=torch.bfloat16, device="cuda")
    dE = torch.zeros(V, h, dtype=torch.float32, device="cuda")
    nws = L.tp_vocab_embedding_backward_workspace_size(N)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    fwd = lambda: (flush.zero_(), L.tp_vocab_embedding_forward(ids, N, V, h, t, inp["E"], Y))
    bwd = lambda: (flush.zero_(), L.tp_vocab_embedding_backward(ids, inp["dY"], N, V, h, t, dE, 1, ws, nws))
    fl_ms = _time(torch, flush.zero_, 10)
    f_ms = _time(torch, fwd, 20) - fl_ms
    b_ms = _time(torch, bwd, 20) - fl_ms
    uniq = int(torch.unique(ids).numel())
    fwd_bytes = 2 * N * h * 2
    bwd_bytes = N * h * 2 + 2 * uniq * h * 4
    hbm = measured_peaks()["hbm"]
    return {"workload": f"vocab-parallel embedding, V={V}, h={h}, t={t}, N={N} Zipf(1.1) token ids ({uniq} distinct)",
            "l2": "256 MB buffer written between calls (flush)",
            "fwd_us": round(f_ms * 1e3, 2), "fwd_GBps": round(fwd_bytes / f_ms / 1e6, 1),
            "fwd_frac_of_hbm": round(fwd_bytes / f_ms / 1e6 / hbm, 4),
            "bwd_us": round(b_ms * 1e3, 2), "bwd_GBps": round(bwd_bytes / b_ms / 1e6, 1),
            "bwd_frac_of_hbm": round(bwd_bytes / b_ms / 1e6 / hbm, 4), "bwd_mode": "accumulate into dE"}


def run_overlap_extra(L, torch, args):
    """Row-parallel GEMM of the TP-MLP (t = 4, A 4 x 2048 x 4096, W_down 16384 x 4096)
    with the g reduction (a) fused into the accumulator, (b) run after the GEMM
    over materialised partials, (c) overlapped tile by tile with the GEMM."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    c = I.CONFIGS["c2"]
    M, h, F, t = c["M"], c["h"], c["F"], c["t"]
    inp = I.mlp_inputs(M, h, F, bias=True, dy=False, seed=0, device="cuda")
    Wdn = torch.empty(t, h, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_row(inp["W_down"], F, h, t, Wdn)
    A = (torch.randn(t, M, F // t, device="cuda") * 0.5).to(torch.bfloat16)
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(t, M, h, dtype=torch.float32, device="cuda")
    nws = L.tp_row_parallel_overlap_workspace_size(M, F, h, t)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    nsk = L.tp_row_parallel_workspace_size(M, F, h, t)
    skws = torch.empty(nsk, dtype=torch.uint8, device="cuda")
    fused = lambda: L.tp_row_parallel_forward(A, M, F, h, t, Wdn, inp["b_down"], None, Y)
    fused_sk = lambda: L.tp_row_parallel_forward_ws(A, M, F, h, t, Wdn, inp["b_down"], None, Y, skws, nsk)

    ovl = lambda: L.tp_row_parallel_forward_overlap(A, M, F, h, t, Wdn, inp["b_down"], None, Y, None, ws, nws)
    iters = max(10, min(args.steps, 30))
    f_ms = _time(torch, fused, iters)
    fsk_ms = _time(torch, fused_sk, iters)
    o_ms = _time(torch, ovl, iters)
    # whole MLP forward in the three modes: the difference to the column-parallel half is the row part
    Wup = torch.empty(t, F // t, h, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_col(inp["W_up"], h, F, t, Wup)
    Aout = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
    act = L.ACT_BY_NAME["gelu_tanh"]
    col = lambda: L.tp_column_parallel_forward(inp["X"], M, h, F, t, act, Wup, inp["b_up"], None, Aout)
    c_ms = _time(torch, col, iters)
    mode_ms = {}
    for name, flag in (("fused", 0), ("unfused", L.TP_FLAG_UNFUSED_REDUCE), ("overlap", L.TP_FLAG_OVERLAP_REDUCE)):
        nw = L.tp_mlp_workspace_size(M, h, F, t, flag)
        w2 = torch.empty(max(nw, 256), dtype=torch.uint8, device="cuda")
        run = lambda: L.tp_mlp_forward(inp["X"], M, h, F, t, act, Wup, inp["b_up"], Wdn, inp["b_down"], None, Y,
                                       None, Aout, flag, w2, w2.numel())
        mode_ms[name] = _time(torch, run, iters) - c_ms
        del w2
    # unfused through the MLP entry's flag needs the column-parallel half too: time it as
    # the overlapped GEMM's partial writes plus the standalone reduction kernel
    red = lambda: L.tp_shard_reduce(P, M, h, t, inp["b_down"], None, Y, None)
    r_ms = _time(torch, red, iters)
    flops = 2.0 * M * h * F
    return {"workload": "row-parallel GEMM + g, t=4, A 4x2048x4096, W_down 16384x4096 (TP-MLP)",
            "fused_ms": round(f_ms, 4), "fused_TFLOPs": round(flops / f_ms / 1e9, 1),
            "fused_splitk_ms": round(fsk_ms, 4), "fused_splitk_TFLOPs": round(flops / fsk_ms / 1e9, 1),
            "overlap_ms": round(o_ms, 4), "overlap_TFLOPs": round(flops / o_ms / 1e9, 1),
            "separate_reduce_kernel_ms": round(r_ms, 4),
            "gemm_plus_reduce_ms": round(mode_ms["unfused"], 4),
            "row_part_in_mlp_forward_ms": {k: round(v, 4) for k, v in mode_ms.items()},
            "partial_bytes": t * M * h * 4,
            "note": "overlap = every shard's fp32 partial tile written, and each tile's shards summed "
                    "inside the GEMM while later tiles compute (tp-comm-overlap stand-in); "
                    "row_part_in_mlp_forward_ms['unfused'] is the GEMM writing partials plus the "
                    "separate reduction kernel"}


def run_mlp_fwd_extra(L, torch, args):
    """The forward-only MLP workload: t = 2, X 128x1024, 1024 -> 4096 -> 1024."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    from megatron_tensor_transformer_shard_gb300 import tp as T
    c = I.CONFIGS["c1"]
    M, h, F, t = c["M"], c["h"], c["F"], c["t"]
    inp = I.mlp_inputs(M, h, F, bias=True, dy=False, seed=0, device="cuda")
    w = T.MLPWeights(inp["W_up"], inp["b_up"], inp["W_down"], inp["b_down"], t)
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
    act = L.ACT_BY_NAME["gelu_tanh"]
    fwd = lambda: L.tp_mlp_forward(inp["X"], M, h, F, t, act, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A,
                                   0, None, 0)
    ms = _time(torch, fwd, max(50, args.steps), warmup=10)
    # The same forward replayed from a CUDA graph: no host work (argument checks, tensor-map
    # encoding, launches) between the kernels; this size is launch-bound otherwise.
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        fwd()
        with torch.cuda.graph(graph, stream=cs):
            fwd()
    torch.cuda.current_stream().wait_stream(cs)
    ms_graph = _time(torch, graph.replay, max(50, args.steps), warmup=10)
    fl = 4.0 * M * h * F
    return {"workload": "TP-MLP forward, t=2, X 128x1024, W_up 1024x4096, W_down 4096x1024, GeLU(tanh)",
            "us_per_step": round(ms * 1e3, 2), "TFLOPs": round(fl / (ms / 1e3) / 1e12, 2),
            "us_per_step_graph": round(ms_graph * 1e3, 2), "TFLOPs_graph": round(fl / (ms_graph / 1e3) / 1e12, 2),
            "flops_per_step": fl, "l2": "8.4 MB of weights stay in L2 (no flush): latency-bound, 32 + 16 tiles",
            "page_bytes": {"expanded_tensor": M * F * 2, "output_reduction_tensor": M * h * 2}}


def run_swiglu_extra(L, torch, args):
    """Token-parallel SwiGLU MLP fwd+bwd at decode-config weight shapes (Llama-3-70B-sized, t = 4)
    over 2048 tokens: column-parallel GEMM over the interleaved gate / up weights with silu(gate) * up
    in its epilogue, row-parallel GEMM + g; backward: the dgrad GEMM whose epilogue forms the gate / up
    gradient, both wgrads and the f sum."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    from megatron_tensor_transformer_shard_gb300 import tp as T
    M, h, F, t = 2048, 8192, 28672, 4
    inp = I.swiglu_inputs(M, h, F, seed=0, device="cuda", dy=True)
    w = T.SwiGLUWeights(inp["W_gate"], inp["W_up"], inp["W_down"], None, t)
    del inp["W_gate"], inp["W_up"], inp["W_down"]
    X, dY = inp["X"], inp["dY"]
    Y, Z, A = T.mlp_forward(X, w, "swiglu")
    grads = T.mlp_backward(dY, X, Z, A, w, "swiglu")
    nws_f = L.tp_mlp_workspace_size(M, h, F, t, 0)
    nws_b = L.tp_mlp_backward_workspace_size(M, h, F, t, 0)
    wsb = torch.empty(nws_b, dtype=torch.uint8, device="cuda")
    wsf = torch.empty(nws_f, dtype=torch.uint8, device="cuda")
    act = L.ACT_BY_NAME["swiglu"]
    dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")

    def step():
        L.tp_mlp_forward(X, M, h, F, t, act, w.Wup_p, None, w.Wdown_p, None, None, Y, Z, A, 0, wsf, nws_f)
        L.tp_mlp_backward(dY, X, Z, A, M, h, F, t, act, w.Wup_p, w.Wdown_p, dX, grads["dWup_p"], grads["dWdown_p"],
                          None, grads["dbdown"], 0, 0, wsb, nws_b)
    ms = _time(torch, step, max(5, min(args.steps, 10)))
    fl = 18.0 * M * h * F  # forward 6 M h F (gate + up + down), backward twice that
    return {"workload": f"SwiGLU MLP fwd+bwd, t={t}, X {M}x{h}, W_gate/W_up {h}x{F}, W_down {F}x{h}",
            "ms_per_step": round(ms, 3), "TFLOPs": round(fl / (ms / 1e3) / 1e12, 1), "flops_per_step": fl,
            "note": "silu(gate) * up and its gradient are computed in the GEMM epilogues"}


def run_attn_extra(L, torch, args, name="c5"):
    """Head-sharded attention block alone at a layer config's shapes: QKV
    column-parallel GEMM, per-head causal flash attention, W_o row-parallel
    GEMM + g; forward and backward."""
    import math
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    from megatron_tensor_transformer_shard_gb300 import tp as T
    c = I.CONFIGS[name]
    N, d, t, nh, dh = c["N"], c["d"], c["t"], c["n_heads"], c["head_dim"]
    inp = I.attn_inputs(N, d, bias=True, dy=True, seed=0, device="cuda")
    bf16, f32 = torch.bfloat16, torch.float32
    Wqkv = torch.empty(t, 3 * d // t, d, dtype=bf16, device="cuda")
    bqkv = torch.empty(t, 3 * d // t, dtype=bf16, device="cuda")
    Wo = torch.empty(t, d, d // t, dtype=bf16, device="cuda")
    L.tp_pack_qkv_heads(inp["W_qkv"], d, nh, dh, t, Wqkv)
    L.tp_pack_qkv_bias(inp["b_qkv"], d, nh, dh, t, bqkv)
    L.tp_pack_row(inp["W_o"], d, d, t, Wo)
    del inp["W_qkv"], inp["W_o"]
    Y = torch.empty(N, d, dtype=bf16, device="cuda")
    QKV = torch.empty(t, N, 3 * d // t, dtype=torch.float16, device="cuda")
    O = torch.empty(t, N, d // t, dtype=bf16, device="cuda")
    lse = torch.empty(t, nh // t, N, dtype=f32, device="cuda")
    sc = 1.0 / math.sqrt(dh)
    naw = L.tp_attn_forward_workspace_size(N, d, nh, dh, t, 0)
    aws = torch.empty(naw, dtype=torch.uint8, device="cuda")
    fwd = lambda: L.tp_attn_forward(inp["X"], N, d, nh, dh, t, 1, sc, Wqkv, bqkv, Wo, inp["b_o"], None, Y, QKV, O,
                                    lse, 0, aws, naw)
    f_ms = _time(torch, fwd, max(5, min(args.steps, 20)))
    dX = torch.empty(N, d, dtype=bf16, device="cuda")
    gq = torch.empty(t, 3 * d // t, d, dtype=f32, device="cuda")
    gbq = torch.empty(t, 3 * d // t, dtype=f32, device="cuda")
    go = torch.empty(t, d, d // t, dtype=f32, device="cuda")
    gbo = torch.empty(d, dtype=f32, device="cuda")
    nws = L.tp_attn_backward_workspace_size(N, d, nh, dh, t, 0)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    bwd = lambda: L.tp_attn_backward(inp["dY"], inp["X"], QKV, O, lse, N, d, nh, dh, t, 1, sc, Wqkv, Wo, dX, gq, gbq,
                                     go, gbo, 0, 0, ws, nws)
    b_ms = _time(torch, bwd, max(5, min(args.steps, 20)))
    # The attention core alone (one forward kernel; the backward's three kernels) on the block's own QKV.
    dO = torch.randn(t, N, d // t, device="cuda").to(torch.float16)
    Dvec = torch.empty(t, nh // t, N, dtype=f32, device="cuda")
    dQKV = torch.empty(t, N, 3 * d // t, dtype=bf16, device="cuda")
    cf_ms = _time(torch, lambda: L.tp_attn_core_forward(QKV, N, d, nh, nh, dh, t, 1, sc, O, lse),
                  max(5, min(args.steps, 20)))
    cb_ms = _time(torch, lambda: L.tp_attn_core_backward(QKV, O, dO, lse, N, d, nh, nh, dh, t, 1, sc, Dvec, dQKV),
                  max(5, min(args.steps, 20)))
    proj = 2.0 * N * d * 3 * d + 2.0 * N * d * d
    core = 2.0 * N * N * d  # causal: QK^T and PV over the unmasked half
    core_bwd = 2.0 * core   # dV, dP, dQ, dK (the recomputed S counted as the forward's)
    return {"workload": f"attention block, t={t}, N={N}, d={d}, {nh} heads x {dh}, causal",
            "fwd_ms": round(f_ms, 3), "fwd_TFLOPs": round((proj + core) / (f_ms / 1e3) / 1e12, 1),
            "bwd_ms": round(b_ms, 3), "bwd_TFLOPs": round(2 * (proj + core) / (b_ms / 1e3) / 1e12, 1),
            "flops_fwd": proj + core, "flops_core_fwd": core,
            "core_fwd_ms": round(cf_ms, 4), "core_fwd_TFLOPs": round(core / (cf_ms / 1e3) / 1e12, 1),
            "core_bwd_ms": round(cb_ms, 4), "core_bwd_TFLOPs": round(core_bwd / (cb_ms / 1e3) / 1e12, 1),
            "core_note": "core FLOPs count the unmasked half only: forward 2*N^2*d (QK^T, PV), backward twice that"}


def run_ln_extra(L, torch, args, name="c5"):
    """Sequence-parallel LayerNorm kernels alone (HBM-bound) at a layer config's shape."""
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    c = I.CONFIGS[name]
    s, h, t = c["N"], c["d"], c["t"]
    inp = I.ln_inputs(s, h, seed=0, device="cuda")
    Xn = torch.empty(s, h, dtype=torch.bfloat16, device="cuda")
    mean = torch.empty(s, dtype=torch.float32, device="cuda")
    rstd = torch.empty(s, dtype=torch.float32, device="cuda")
    # inputs of 64 MB stay partly in the 129 MB L2 between launches: flush it between timed calls
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    X = inp["X"]

    def fwd():
        flush.zero_()
        L.tp_sp_layernorm_forward(X, s, h, t, inp["gamma"], inp["beta"], 1e-5, Xn, mean, rstd)

    dX = torch.empty(s, h, dtype=torch.bfloat16, device="cuda")
    parts = [torch.empty(t, h, dtype=torch.float32, device="cuda") for _ in range(2)]
    dg, db = (torch.empty(h, dtype=torch.float32, device="cuda") for _ in range(2))

    def bwd():
        flush.zero_()
        L.tp_sp_layernorm_backward(inp["dY"], X, inp["gamma"], mean, rstd, X, s, h, t, dX, parts[0], parts[1], dg, db)

    fl_ms = _time(torch, flush.zero_, 10)
    f_ms = _time(torch, fwd, 20) - fl_ms
    b_ms = _time(torch, bwd, 20) - fl_ms
    fwd_bytes = 2 * s * h * 2 + 2 * h * 2 + 2 * s * 4
    bwd_bytes = 6 * s * h * 2 + s * 8 + 2 * t * h * 4 * 2
    hbm = measured_peaks()["hbm"]
    return {"workload": f"SP LayerNorm, [{t}][{s // t}][{h}]", "l2": "256 MB buffer written between calls (flush)",
            "fwd_us": round(f_ms * 1e3, 2), "fwd_GBps": round(fwd_bytes / f_ms / 1e6, 1),
            "fwd_frac_of_hbm": round(fwd_bytes / f_ms / 1e6 / hbm, 4),
            "bwd_us": round(b_ms * 1e3, 2), "bwd_GBps": round(bwd_bytes / b_ms / 1e6, 1),
            "bwd_frac_of_hbm": round(bwd_bytes / b_ms / 1e6 / hbm, 4)}


def layer_flops(N, d, F):
    """fwd = QKV + W_o + MLP GEMMs + causal attention (unmasked half); fwd+bwd = 3 x fwd."""
    fwd = 2.0 * N * d * 3 * d + 2.0 * N * d * d + 4.0 * N * d * F + 2.0 * N * N * d
    return 3.0 * fwd


def run_layer_extra(L, torch, args, name):
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    from megatron_tensor_transformer_shard_gb300 import tp as T
    c = I.CONFIGS[name]
    N, d, F, t, nh, sp = c["N"], c["d"], c["F"], c["t"], c["n_heads"], c["sp"]
    inp = I.layer_inputs(N, d, F, seed=0, device="cuda")
    w = T.LayerWeights(inp, nh, c["head_dim"], t)
    for k in ("W_qkv", "W_o", "W_up", "W_down"):
        del inp[k]
    X, G = inp["X"], inp["dY"]

    def step():
        Y, saved = T.layer_forward(X, w, sp=sp)
        T.layer_backward(G, saved, w)

    ms = _time(torch, step, max(5, min(args.steps, 20)), warmup=3)
    fl = layer_flops(N, d, F)
    peak = measured_peaks()["bf16_burst"]
    out = {"workload": (f"{'sequence-parallel ' if sp else ''}TP layer fwd+bwd, t={t}, N={N}, d={d}, "
                        f"{nh} heads x {c['head_dim']}, MLP {d}->{F}, causal"),
           "ms_per_step": round(ms, 3), "TFLOPs": round(fl / (ms / 1e3) / 1e12, 1), "flops_per_step": fl,
           "frac_of_peak": round(fl / (ms / 1e3) / 1e12 / peak, 4)}
    del w, inp
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------- oracle (CPU)

def _f64(O, I, v):
    return O.bf16_to_f64(I.bits(v)).reshape(tuple(v.shape))


def _oracle_inputs(M_s, seed=0, return_cpu=False):
    import oracle as O
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    cfg = I.CONFIGS[WORKLOAD]
    inp = I.mlp_inputs(cfg["M"], cfg["h"], cfg["F"], bias=True, dy=True, seed=seed)
    r = {k: _f64(O, I, v) for k, v in inp.items()}
    r["X"], r["dY"] = r["X"][:M_s], r["dY"][:M_s]
    return (r, cfg, inp) if return_cpu else (r, cfg)


def _oracle_step(O, r, cfg):
    f = O.mlp_forward_sharded(r["X"], r["W_up"], r["b_up"], r["W_down"], r["b_down"], cfg["act"], cfg["t"])
    b = O.mlp_backward_sharded(r["dY"], r["X"], r["W_up"], r["W_down"], f, cfg["act"], cfg["t"])
    return f, b


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _timed(fn):
    t0 = time.perf_counter()
    out = fn()
    return time.perf_counter() - t0, out


def _rel(gpu, ref):
    import numpy as np
    return float(np.abs(gpu - ref).max() / max(np.abs(ref).max(), 1e-30))


def oracle_probe(name, rows=0):
    """Seconds of the fp64 oracle, as it stands, on one configuration (or a stated
    sample of it); inputs are drawn first and not timed."""
    import oracle as O
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    if name == "c1":
        c = I.CONFIGS["c1"]
        inp = I.mlp_inputs(c["M"], c["h"], c["F"], bias=True, dy=False, seed=0)
        r = {k: _f64(O, I, v) for k, v in inp.items() if v is not None}
        sec, _ = _timed(lambda: O.mlp_forward_sharded(r["X"], r["W_up"], r["b_up"], r["W_down"], r["b_down"],
                                                      c["act"], c["t"]))
        return {"seconds": sec, "sample": "the whole forward (128 tokens)", "scale": 1.0}
    if name == "c2":
        r, cfg = _oracle_inputs(rows)
        sec, _ = _timed(lambda: _oracle_step(O, r, cfg))
        return {"seconds": sec, "sample": f"fwd+bwd on the first {rows} of {cfg['M']} token rows",
                "scale": cfg["M"] / rows}
    if name == "c3":
        # one shard's slice of the decode MLP (7168 of 28672 hidden units): the loop body of the
        # sharded oracle for shard 0; the whole step is t such slices
        c = I.CONFIGS["c3"]
        Ft = c["F"] // c["t"]
        inp = I.swiglu_inputs(c["M"], c["h"], Ft, seed=0)
        r = {k: _f64(O, I, v) for k, v in inp.items()}
        sec, _ = _timed(lambda: O.swiglu_forward_sharded(r["X"], r["W_gate"], r["W_up"], r["W_down"], 1))
        return {"seconds": sec, "sample": f"shard 0's slice ({Ft} of {c['F']} hidden units), x{c['t']}",
                "scale": float(c["t"])}
    # c4 / c5: the whole layer's weights, forward + backward on a prefix of the tokens (causal
    # attention of a prefix depends on the prefix only)
    import math
    c = I.CONFIGS[name]
    d, F, t, nh = c["d"], c["F"], c["t"], c["n_heads"]
    inp = I.layer_inputs(rows, d, F, seed=0)
    r = {k: _f64(O, I, v) for k, v in inp.items()}
    del inp
    cfg = {"n_heads": nh, "head_dim": c["head_dim"], "causal": True, "scale": 1.0 / math.sqrt(c["head_dim"]),
           "eps": c["eps"], "act": c["act"]}
    p = {k: v for k, v in r.items() if k not in ("X", "dY")}
    X, G = r["X"], r["dY"]
    if c["sp"]:
        X, G = X.reshape(t, rows // t, d), G.reshape(t, rows // t, d)

    def step():
        f = O.layer_forward(X, p, cfg, t, c["sp"])
        O.layer_backward(G, X, p, cfg, t, f, c["sp"])
    sec, _ = _timed(step)
    return {"seconds": sec, "sample": f"fwd+bwd on the first {rows} of {c['N']} tokens, all weights",
            "scale": None}


def _probe_subprocess(name, rows, threads):
    """oracle_probe in a fresh interpreter whose BLAS and OpenMP use `threads` threads."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe", name, "--probe-rows", str(rows)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc={r.returncode}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def _host_mem_available_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 2 ** 20
    except OSError:
        pass
    return None


def cpu_baseline(budget_s=12.0, gpu=None, layers=False, per_config=True):
    """The fp64 oracle as it stands, timed on the host cores: on a row sample of the
    headline workload sized to about `budget_s` seconds (the baseline value), and per
    configuration (all cores, and single-threaded for the two MLP workloads).  With
    `gpu`, the same path that was timed also runs on the host-drawn inputs and its
    rows are compared with the oracle's: max|gpu - oracle| / max|oracle| per output."""
    import oracle as O
    from megatron_tensor_transformer_shard_gb300 import inputs as I
    r, cfg = _oracle_inputs(cfg_rows := 128)
    dt, _ = _timed(lambda: _oracle_step(O, r, cfg))
    rows = int(min(cfg["M"], max(128, (budget_s / max(dt, 1e-3)) * 128 // 128 * 128)))
    r, cfg, inp = _oracle_inputs(rows, return_cpu=True)
    dt, (f, b) = _timed(lambda: _oracle_step(O, r, cfg))
    fl = flops_per_step(rows, cfg["h"], cfg["F"])
    cores = _cores()
    out = {"value": round(fl / dt / 1e12, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"one fwd+bwd of the same MLP on the first {rows} of {cfg['M']} token rows "
                     f"(numpy fp64, {dt:.2f} s)", "seconds": round(dt, 3)}
    parity = None
    if gpu is not None:
        g = gpu.run(inp, cfg["M"], cfg["h"], cfg["F"], cfg["t"], cfg["act"], backward=True)
        parity = {"c2": {"rows": rows, "Y": round(_rel(_f64(O, I, g["Y"])[:rows], f["Y"]), 6),
                         "dX": round(_rel(_f64(O, I, g["dX"])[:rows], b["dX"]), 6)}}
        c1 = I.CONFIGS["c1"]
        inp1 = I.mlp_inputs(c1["M"], c1["h"], c1["F"], bias=True, dy=False, seed=0)
        r1 = {k: _f64(O, I, v) for k, v in inp1.items() if v is not None}
        f1 = O.mlp_forward_sharded(r1["X"], r1["W_up"], r1["b_up"], r1["W_down"], r1["b_down"], c1["act"], c1["t"])
        g1 = gpu.run(inp1, c1["M"], c1["h"], c1["F"], c1["t"], c1["act"], backward=False)
        parity["c1"] = {"rows": c1["M"], "Y": round(_rel(_f64(O, I, g1["Y"]), f1["Y"]), 6)}
        parity["bound"] = 1e-2
    del r, inp, f, b
    if not per_config:
        return out, parity
    per = {}
    probes = [("c1", 0), ("c3", 0)]
    # The layer probes hold the whole layer's weights and weight gradients in fp64 on the
    # host (C5 ~13 GB, C4 ~30 GB): C5 runs when the host has room, C4 only when asked.
    avail = _host_mem_available_gb()
    for name, need_gb in (("c5", 40.0), ("c4", 90.0)):
        if (name == "c5" or layers) and avail is not None and avail >= need_gb:
            probes.append((name, 32))
        else:
            per[name] = {"skipped": f"needs --cpu-layers and ~{need_gb:.0f} GB of free host memory "
                                    f"({avail if avail is None else round(avail)} GB free)"
                         if name == "c4" else f"needs ~{need_gb:.0f} GB of free host memory ({avail} GB free)"}
    for name, rows_p in probes:
        try:
            pr = oracle_probe(name, rows_p)
            per[name] = {"seconds": round(pr["seconds"], 3), "cores": cores, "sample": pr["sample"]}
            if pr.get("scale"):
                per[name]["seconds_whole_config"] = round(pr["seconds"] * pr["scale"], 3)
        except Exception as e:  # reported, not fatal: the headline baseline stands
            per[name] = {"error": f"{type(e).__name__}: {e}"[:160]}
    for name, rows_p in (("c1", 0), ("c2", 64)):
        pr = _probe_subprocess(name, rows_p, 1)
        if "seconds" in pr:
            per[name + "_1thread"] = {"seconds": round(pr["seconds"], 3), "cores": 1, "sample": pr["sample"]}
            if pr.get("scale"):
                per[name + "_1thread"]["seconds_whole_config"] = round(pr["seconds"] * pr["scale"], 3)
        else:
            per[name + "_1thread"] = pr
    out["per_config"] = per
    return out, parity


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle as O
    rows = args.reference_rows
    r, cfg = _oracle_inputs(rows)
    for _ in range(args.warmup):
        _oracle_step(O, r, cfg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(O, r, cfg)
    dt = (time.perf_counter() - t0) / args.steps
    value = flops_per_step(rows, cfg["h"], cfg["F"]) / dt / 1e12
    sample = f"each step one fwd+bwd of the same MLP on the first {rows} of {cfg['M']} token rows (numpy fp64)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "TP-MLP fwd+bwd, t=4, X 2048x4096, W_up 4096x16384, W_down 16384x4096, "
                                   "GeLU(tanh)", "global_batch": rows, "seq_len": rows,
                       "parallelism": "t=4 logical shards (oracle loop)"},
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_only(args):
    import torch
    torch.cuda.set_device(dist_env()[2])
    from megatron_tensor_transformer_shard_gb300 import build as B
    B.build()
    from megatron_tensor_transformer_shard_gb300 import _lib as L
    if args.only == "c1":
        return {"mlp_fwd_c1": run_mlp_fwd_extra(L, torch, args)}
    if args.only == "c3":
        return {"decode_c3": run_decode_extra(L, torch, args)}
    if args.only == "attn":
        return {"attention_c5": run_attn_extra(L, torch, args)}
    if args.only == "ln":
        return {"sp_layernorm_c5": run_ln_extra(L, torch, args)}
    if args.only == "dattn":
        return {"decode_attention": run_decode_attn_extra(L, torch, args)}
    if args.only == "emb":
        return {"vocab_embedding": run_embedding_extra(L, torch, args)}
    if args.only == "swiglu":
        return {"swiglu_mlp": run_swiglu_extra(L, torch, args)}
    if args.only == "ovl":
        return {"row_parallel_overlap_c2": run_overlap_extra(L, torch, args)}
    return {f"layer_{args.only}": run_layer_extra(L, torch, args, args.only)}


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--cpu-layers", action="store_true",
                   help="also time the oracle on the 2048-token layer (32-token prefix; ~30 GB of host memory)")
    p.add_argument("--reference-rows", type=int, default=64, help="token rows per oracle step (--impl reference)")
    p.add_argument("--oracle-probe", choices=["c1", "c2", "c3", "c4", "c5"], default=None,
                   help=argparse.SUPPRESS)  # one timed oracle run (used by the single-thread baseline)
    p.add_argument("--probe-rows", type=int, default=64, help=argparse.SUPPRESS)
    p.add_argument("--only", choices=["c1", "c3", "c4", "c5", "attn", "ln", "dattn", "emb", "ovl", "swiglu"], default=None,
                   help="run only one secondary workload (forward MLP c1, decode c3, layers c4/c5, the c5-shaped "
                        "attention block, SP LayerNorm, decode attention over a sharded KV cache, the "
                        "vocab-parallel embedding or the overlapped row-parallel reduction) and print it")
    args = p.parse_args()
    if args.oracle_probe:
        print(json.dumps(oracle_probe(args.oracle_probe, args.probe_rows)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.only:
        print(json.dumps(run_only(args)), flush=True)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
