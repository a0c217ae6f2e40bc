#!/usr/bin/env python
"""Benchmark of one training step of the head-chunked attention layer.

One step = upipe_attn_fwd + upipe_attn_bwd of a GQA/RoPE causal attention
layer (projections, RoPE, attention, output projection; forward and
backward with per-chunk recomputation) on synthetic bf16 inputs resident in
HBM.  Default workload: the 32B-shaped layer (L=131072, D=5120, H=64, Hkv=8,
d=128) with U=8 query heads per chunk.

Prints one JSON line.  `value` is the layer's algorithmic TFLOP/s (causal
attention fwd+bwd 7*L^2*H*d plus the projections' 3*(2*L*D*(H+2Hkv)*d +
2*L*H*d*D); the backward recomputation is hardware work and is not counted)
over the device-timed steps, which run with per-launch timing off; a
separate profiled step gives the per-kernel table, the attention-only
figure and the roofline.  A U sweep measures each chunk size's workspace
high-water mark on the device next to the library's own arithmetic.
`--impl reference` times the fp64 CPU oracle on the same metric instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import socket
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal attn fwd+bwd TFLOP/s (% BF16 peak) at 1 GB300; peak activation bytes vs U"

WORKLOADS = {
    "qwen32b_layer_L131072_U8": dict(L=131072, D=5120, H=64, Hkv=8, U=8),
    "llama3_8b_layer_L32768_U8": dict(L=32768, D=4096, H=32, Hkv=8, U=8),
    "tiny_L1024_U2": dict(L=1024, D=1024, H=8, Hkv=2, U=2),
    "llama3_8b_layer_L65536_U4": dict(L=65536, D=4096, H=32, Hkv=8, U=4),
    "llama3_8b_layer_L262144_U4": dict(L=262144, D=4096, H=32, Hkv=8, U=4),
}
DEFAULT = "qwen32b_layer_L131072_U8"
# Chunk sizes measured by the U sweep (the workload's U among them).
U_SWEEP = {
    "qwen32b_layer_L131072_U8": (64, 16, 8),
    "llama3_8b_layer_L32768_U8": (32, 8, 4),
    "tiny_L1024_U2": (8, 4, 2),
    "llama3_8b_layer_L65536_U4": (32, 8, 4),
    "llama3_8b_layer_L262144_U4": (32, 8, 4),
}
# The MLP and vocabulary of the model family each workload's layer belongs
# to (Llama-3-8B: F = 14336, V = 128256; Qwen2.5-32B: F = 27648, V = 152064),
# for the sequence-tiled MLP and loss measured beside the layer; T rows per
# tile.
ALST_SHAPES = {
    "qwen32b_layer_L131072_U8": dict(F=27648, V=152064, T_mlp=8192, T_ce=4096),
    "llama3_8b_layer_L32768_U8": dict(F=14336, V=128256, T_mlp=8192, T_ce=4096),
    "tiny_L1024_U2": dict(F=2048, V=4096, T_mlp=256, T_ce=256),
    "llama3_8b_layer_L65536_U4": dict(F=14336, V=128256, T_mlp=8192, T_ce=4096),
    "llama3_8b_layer_L262144_U4": dict(F=14336, V=128256, T_mlp=8192, T_ce=4096),
}
TARGET_FRAC_OF_BURST = 0.55
O_MODE_NOTE = {
    "host": "kept in page-locked host memory: each chunk's O copied out during the forward and back during "
            "the backward on copy streams, inside the timed step; the backward does not recompute it",
    "recompute": "recomputed by the backward from the forward's LSE (a second pass over the keys)",
}
# Kernel kinds that are not attention: they run one at a time on the
# caller's stream, so their event times add up to the step's projection time.
PROJ_KINDS = ("rope_table", "qkv_gemm", "oproj_gemm", "do_gemm", "dwo_gemm", "dwqkv_gemm", "dx_gemm", "delta",
              "zero_rows")


def layer_flops(L, D, H, Hkv, d=128):
    attn = 7.0 * L * L * H * d
    proj = 3.0 * (2.0 * L * D * (H + 2 * Hkv) * d + 2.0 * L * H * d * D)
    return attn, proj


def kernel_flops(kind, w, d=128):
    """Algorithmic flops of one launch of `kind` in the layer path."""
    L, D, H, Hkv, U = w["L"], w["D"], w["H"], w["Hkv"], w["U"]
    g = H // Hkv
    kvc = U // g if U >= g else 1
    slots = U + 2 * kvc
    tri = L * L / 2.0  # causal (query, key) pairs per head
    return {
        "attn_fwd": 2 * 2 * tri * U * d,        # S = QK^T, O = PV
        "attn_bwd_dkdv": 4 * 2 * tri * U * d,   # S^T, dP^T, dV, dK
        "attn_bwd_dq": 3 * 2 * tri * U * d,     # S, dP, dQ
        "qkv_gemm": 2.0 * L * slots * d * D,
        "oproj_gemm": 2.0 * L * U * d * D,
        "do_gemm": 2.0 * L * U * d * D,
        "dwo_gemm": 2.0 * L * U * d * D,
        "dwqkv_gemm": 2 * 2.0 * L * slots * d * D,  # high and low halves
        "dx_gemm": 2 * 2.0 * L * slots * d * D,
    }.get(kind)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return m.get("bf16_tflops", 1900.0), m.get("bf16_tflops_sustained", 1700.0), m.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_sample(L):
    """Times the fp64 oracle on one query head (H = Hkv = 1) of causal
    attention fwd+bwd at sequence length L; returns (TFLOP/s, seconds)."""
    import numpy as np
    from headwise_chunked_context_gb300 import synth
    from oracle import upipe_oracle as orc
    q, k, v, do = synth.core_inputs(L, 1, 1)
    q, k, v, do = (t.double().numpy() for t in (q, k, v, do))
    t0 = time.perf_counter()
    o, lse = orc.attention_core_fwd(q, k, v)
    orc.attention_core_bwd(q, k, v, o, lse, do)
    dt = time.perf_counter() - t0
    return 7.0 * L * L * 128 / dt / 1e12, dt


def max_over_ranks(value: float, device) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flops_per_step_per_rank / (ms_per_step / 1e3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    L_sample = args.ref_sample_L
    for _ in range(args.warmup):
        cpu_oracle_sample(L_sample)
    vals, secs = [], []
    for _ in range(args.steps):
        v, s = cpu_oracle_sample(L_sample)
        vals.append(v)
        secs.append(s)
    value = statistics.mean(vals)
    cores = os.cpu_count()
    sample = (f"fp64 NumPy oracle, one query head (H=Hkv=1, d=128) of causal attention fwd+bwd at "
              f"L={L_sample} per step, standing in for the {args.workload} workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **w},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def strip_comments(text):
    """C/C++ source without its comments and blank-line noise, so that a
    comment-only edit does not invalidate a stored capture."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_sha(name):
    """Hash of a kernel's source file together with the headers every kernel
    includes (comments removed), so that a change to the code of either
    invalidates a stored capture."""
    h = hashlib.sha256()
    for f in (name, "sm103_ptx.cuh", "upipe_internal.h"):
        with open(os.path.join(ROOT, "headwise_chunked_context_gb300", "csrc", f)) as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


# Kernels launched concurrently with another (value): their event interval
# includes time queued behind it.
OVERLAPPED = {"attn_bwd_dq": "attn_bwd_dkdv"}
KIND_SOURCE = {"attn_fwd": "attn_fwd.cu", "attn_bwd_dq": "attn_bwd.cu", "attn_bwd_dkdv": "attn_bwd.cu"}


def traffic_for(kind, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        t = json.load(f)
    e = t.get(kind)
    if not e or e.get("workload") != workload:
        return None
    src = KIND_SOURCE.get(kind, "gemm.cu")
    if e.get("source_sha") != source_sha(src):
        return None
    return e.get("bytes_per_launch")


def _bytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def alst_section(workload, w, dev, stream, steps=2):
    """The sequence-tiled SwiGLU MLP and LM-head cross-entropy at the
    workload's L and D and its model family's F and V: device-timed forward
    and backward, algorithmic TFLOP/s (MLP: 6 L D F forward, 12 L D F
    backward; loss: 6 L D V), and each call's device high-water mark next
    to the library's workspace for one tile."""
    from headwise_chunked_context_gb300 import synth, upipe
    a = ALST_SHAPES[workload]
    L, D, F, V = w["L"], w["D"], a["F"], a["V"]

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    def peak(fn):
        """Device high-water mark of one allocating call, less its outputs."""
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        out = fn()
        torch.cuda.synchronize(dev)
        return torch.cuda.max_memory_allocated(dev) - base - _bytes(*out)

    T = a["T_mlp"]
    x, wgu, wd, dy = synth.mlp_inputs(L, D, F, device=dev)
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dwgu = torch.empty(wgu.shape, dtype=torch.float32, device=dev)
    dwd = torch.empty(wd.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(upipe.mlp_workspace_bytes(L, D, F, T, 1), dtype=torch.uint8, device=dev)
    fwd_ms = timed(lambda: upipe.mlp_fwd(x, wgu, wd, y, T, ws, stream))
    bwd_ms = timed(lambda: upipe.mlp_bwd(x, wgu, wd, dy, dx, dwgu, dwd, T, ws, stream))
    del ws
    pk_b = peak(lambda: upipe.mlp_backward(x, wgu, wd, dy, T))
    mlp = {"L": L, "D": D, "F": F, "T": T, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
           "fwd_tflops": 6.0 * L * D * F / (fwd_ms / 1e3) / 1e12,
           "bwd_tflops": 12.0 * L * D * F / (bwd_ms / 1e3) / 1e12,
           "tflops": 18.0 * L * D * F / ((fwd_ms + bwd_ms) / 1e3) / 1e12,
           "bwd_workspace_bytes": upipe.mlp_workspace_bytes(L, D, F, T, 1), "bwd_peak_bytes_measured": pk_b,
           "untiled_bwd_workspace_bytes": upipe.mlp_workspace_bytes(L, D, F, L, 1),
           "note": "backward recomputes the gate/up GEMM per tile (not counted)"}
    del x, wgu, wd, dy, y, dx, dwgu, dwd
    torch.cuda.empty_cache()
    T = a["T_ce"]
    h, wv, labels = synth.ce_inputs(L, D, V, device=dev)
    scale = 1.0 / int((labels >= 0).sum())
    loss = torch.empty(L, dtype=torch.float32, device=dev)
    dh = torch.empty_like(h)
    dw = torch.empty(wv.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(upipe.ce_workspace_bytes(L, D, V, T), dtype=torch.uint8, device=dev)
    ce_ms = timed(lambda: upipe.ce_fwd_bwd(h, wv, labels, scale, loss, dh, dw, T, ws, stream))
    # Per-kernel split of one call: the softmax rows are HBM-bound (the fp32
    # logits read twice, dZ written in bf16: 10 bytes per logit).
    upipe.profile_enable(True)
    upipe.ce_fwd_bwd(h, wv, labels, scale, loss, dh, dw, T, ws, stream)
    torch.cuda.synchronize(dev)
    upipe.profile_enable(False)
    prof = upipe.profile_read()
    rows_ms, rows_n = prof["ce_rows"]
    rows_gbs = 10.0 * L * V / (rows_ms / 1e3) / 1e9
    del ws
    pk_c = peak(lambda: upipe.ce_loss(h, wv, labels, scale, T))
    ce = {"L": L, "D": D, "V": V, "T": T, "fwd_bwd_ms": ce_ms, "tflops": 6.0 * L * D * V / (ce_ms / 1e3) / 1e12,
          "workspace_bytes": upipe.ce_workspace_bytes(L, D, V, T), "peak_bytes_measured": pk_c,
          "untiled_workspace_bytes": upipe.ce_workspace_bytes(L, D, V, L),
          "mean_loss": float(loss.sum().item() * scale),
          "kernels_ms": {k: v[0] for k, v in prof.items() if v[1] > 0},
          "rows_roofline": {"bound": "hbm", "achieved": rows_gbs, "peak": peaks()[2], "unit": "GB/s",
                            "frac": rows_gbs / peaks()[2], "launches": rows_n,
                            "bytes": "10 per logit: fp32 logits read twice, bf16 dZ written"}}
    del h, wv, labels, loss, dh, dw
    torch.cuda.empty_cache()
    return {"mlp": mlp, "ce": ce}


def u_sweep(w, u_list, dev, stream, x, wqkv, wo, dout, n_timed=1):
    """For each chunk size U: the workspace high-water mark measured on the
    device around the allocating helpers (torch.cuda.max_memory_allocated
    minus the caller-visible outputs), next to the library's arithmetic
    (chunk bytes scale with U, fixed bytes do not), and the step time."""
    from headwise_chunked_context_gb300 import upipe
    L, D, H, Hkv = w["L"], w["D"], w["H"], w["Hkv"]
    rows = []
    attn_f, proj_f = layer_flops(L, D, H, Hkv)
    for u in u_list:
        cfg = upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=u)
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        out, lse, _ = upipe.layer_forward(cfg, x, wqkv, wo)
        torch.cuda.synchronize(dev)
        fwd_peak = torch.cuda.max_memory_allocated(dev) - base - _bytes(out, lse)
        base2 = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        dx, dw, dwo = upipe.layer_backward(cfg, x, wqkv, wo, dout, lse)
        torch.cuda.synchronize(dev)
        bwd_peak = torch.cuda.max_memory_allocated(dev) - base2 - _bytes(dx, dw, dwo)
        ws = torch.empty(max(upipe.workspace_bytes(cfg, 0), upipe.workspace_bytes(cfg, 1)), dtype=torch.uint8,
                         device=dev)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_timed):
            upipe.attn_fwd(cfg, x, wqkv, wo, out, lse, None, ws, stream)
            upipe.attn_bwd(cfg, x, wqkv, wo, dout, lse, dx, dw, dwo, None, ws, stream)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        ms = a0.elapsed_time(a1) / n_timed
        cf, ff = upipe.activation_bytes(cfg, 0)
        cb, fb = upipe.activation_bytes(cfg, 1)
        rows.append({"U": u, "workspace_fwd_measured": fwd_peak, "workspace_bwd_measured": bwd_peak,
                     "workspace_fwd": upipe.workspace_bytes(cfg, 0), "workspace_bwd": upipe.workspace_bytes(cfg, 1),
                     "chunk_bytes_fwd": cf, "fixed_bytes_fwd": ff, "chunk_bytes_bwd": cb, "fixed_bytes_bwd": fb,
                     "ms_per_step": ms, "tflops": (attn_f + proj_f) / (ms / 1e3) / 1e12})
        del out, lse, dx, dw, dwo, ws
    full = [r for r in rows if r["U"] == H]
    if full:
        for r in rows:
            r["chunk_bytes_bwd_vs_unchunked"] = r["chunk_bytes_bwd"] / full[0]["chunk_bytes_bwd"]
            r["chunk_saving_vs_unchunked"] = 1.0 - r["chunk_bytes_bwd_vs_unchunked"]
    torch.cuda.empty_cache()
    return rows


def run_upipe(args, w, world, rank, local):
    from headwise_chunked_context_gb300 import upipe, build
    if not os.path.exists(upipe.LIB_PATH):
        build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L, D, H, Hkv, U = w["L"], w["D"], w["H"], w["Hkv"], w["U"]
    cfg = upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=U)
    stream = torch.cuda.current_stream(dev)

    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    x = torch.randn((L, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    wqkv = (torch.randn(((H + 2 * Hkv) * 128, D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    wo = (torch.randn((D, H * 128), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    dout = torch.randn((L, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    out = torch.empty((L, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, L), dtype=torch.float32, device=dev)
    dx = torch.empty((L, D), dtype=torch.bfloat16, device=dev)
    dwqkv = torch.empty(((H + 2 * Hkv) * 128, D), dtype=torch.float32, device=dev)
    dwo = torch.empty((D, H * 128), dtype=torch.float32, device=dev)
    # Where O waits between forward and backward: "recompute" (the
    # backward recomputes it from the LSE) or "host" (kept in page-locked
    # host memory, two chunk buffers on the device).  The other mode is
    # timed too and reported beside the line.
    modes = (args.o_mode, "host" if args.o_mode == "recompute" else "recompute")
    o_code = {"recompute": upipe.O_RECOMPUTE, "host": upipe.O_HOST}
    ws_bytes = max(upipe.workspace_bytes(cfg, p, o_mode=o_code[m]) for p in (0, 1) for m in modes)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o_host = upipe.new_host_o(cfg)
    torch.cuda.synchronize(dev)

    def layer_step(mode, bx, bw, bwo, bd, bo, bl, bdx, bdw, bdwo):
        if mode == "host":
            upipe.attn_fwd_host_o(cfg, bx, bw, bwo, bo, bl, o_host, ws, stream)
            upipe.attn_bwd_host_o(cfg, bx, bw, bwo, bd, bl, o_host, bdx, bdw, bdwo, ws, stream)
        else:
            upipe.attn_fwd(cfg, bx, bw, bwo, bo, bl, None, ws, stream)
            upipe.attn_bwd(cfg, bx, bw, bwo, bd, bl, bdx, bdw, bdwo, None, ws, stream)

    def step(mode=args.o_mode):
        layer_step(mode, x, wqkv, wo, dout, out, lse, dx, dwqkv, dwo)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def check_status(when):
        code = upipe.last_device_status(stream)
        if code != 0:
            raise RuntimeError(f"device status {when}: {upipe.strerror(code)}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check_status("after warm-up")

    # ---- timed region: K steps, device events, clocks sampled throughout;
    # no per-launch events are recorded here.
    barrier()
    torch.cuda.synchronize(dev)
    n0 = upipe.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    launches = upipe.launch_count() - n0
    barrier()
    ms = e0.elapsed_time(e1)
    clocks = clk.summary()
    check_status("after the timed steps")
    ms = max_over_ranks(ms, dev)

    # ---- profiled pass (separate from the timing): per-launch event pairs
    # on the launching streams.
    n_prof = max(1, min(args.steps, 2))
    upipe.profile_enable(True)
    for _ in range(n_prof):
        step()
    torch.cuda.synchronize(dev)
    upipe.profile_enable(False)
    prof = upipe.profile_read()
    check_status("after the profiled steps")

    # ---- forward and backward timed separately
    def timed(fn, n):
        fn()
        torch.cuda.synchronize(dev)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        return a0.elapsed_time(a1) / n
    n_split = max(1, min(args.steps, 3))
    if args.o_mode == "host":
        fwd_ms = timed(lambda: upipe.attn_fwd_host_o(cfg, x, wqkv, wo, out, lse, o_host, ws, stream), n_split)
        bwd_ms = timed(lambda: upipe.attn_bwd_host_o(cfg, x, wqkv, wo, dout, lse, o_host, dx, dwqkv, dwo, ws,
                                                     stream), n_split)
    else:
        fwd_ms = timed(lambda: upipe.attn_fwd(cfg, x, wqkv, wo, out, lse, None, ws, stream), n_split)
        bwd_ms = timed(lambda: upipe.attn_bwd(cfg, x, wqkv, wo, dout, lse, dx, dwqkv, dwo, None, ws, stream),
                       n_split)
    check_status("after the fwd/bwd split")
    # The other O mode, same inputs, a few steps.
    other_mode = modes[1]
    other_ms = timed(lambda: step(other_mode), n_split)
    check_status("after the other O mode")

    attn_f, proj_f = layer_flops(L, D, H, Hkv)
    step_flops = attn_f + proj_f
    # Hardware work adds the backward's recompute of the QKV slices and, when
    # O is not kept, of the attention forward (2 of attn_f's 7 parts).
    recompute_flops = (attn_f * 2.0 / 7.0 if args.o_mode == "recompute" else 0.0) + 2.0 * L * D * (H + 2 * Hkv) * 128
    ms_step = ms / args.steps
    value = job_tflops(step_flops, ms_step, world)
    burst, sustained, hbm, peak_src = peaks()

    # ---- per-kernel table and roofline of the dominant kernel, from the
    # profiled pass.  dQ runs concurrently with dK/dV on the caller's stream;
    # its event pair opens at the fork, so its interval also holds the time
    # its CTAs waited behind dK/dV's for SMs: it is reported as an interval.
    busy = {k: v for k, v in prof.items() if v[1] > 0}
    solo = {k: v for k, v in busy.items() if k not in OVERLAPPED}
    dom = max(solo, key=lambda k: solo[k][0])
    dom_ms, dom_n = busy[dom]
    fl = kernel_flops(dom, w)
    achieved = fl / (dom_ms / dom_n / 1e3) / 1e12
    traffic = traffic_for(dom, args.workload)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": sustained, "unit": "TFLOP/s",
                "frac": achieved / sustained, "traffic": traffic, "kernel": dom,
                "peak_kind": f"bf16 sustained ({peak_src}): the kernel is timed inside a long step",
                "frac_of_burst": achieved / burst}
    prof_step_ms = sum(v[0] for k, v in busy.items() if k not in OVERLAPPED) / n_prof
    kernels = {k: {"ms_per_step": v[0] / n_prof, "launches_per_step": v[1] / n_prof,
                   "share_of_step": v[0] / n_prof / ms_step} for k, v in solo.items()}
    for k in kernels:
        f = kernel_flops(k, w)
        if f:
            kernels[k]["tflops"] = f / (busy[k][0] / busy[k][1] / 1e3) / 1e12
    for k, other in OVERLAPPED.items():
        if k in busy:
            kernels[k] = {"interval_ms_per_step": busy[k][0] / n_prof,
                          "launches_per_step": busy[k][1] / n_prof, "concurrent_with": other}
    # Attention alone: the step's time less the projection-side kernels
    # (which run one at a time on the caller's stream).
    proj_ms = sum(busy[k][0] for k in PROJ_KINDS if k in busy) / n_prof
    attn_ms = ms_step - proj_ms
    attention = {"tflops": world * attn_f / (attn_ms / 1e3) / 1e12, "ms_per_step": attn_ms,
                 "flops_per_step": attn_f, "frac_of_burst": attn_f / (attn_ms / 1e3) / 1e12 / burst,
                 "note": "7 L^2 H d over the step time less the projection kernels' event time"}

    # ---- end to end through the public API with host buffers.  Each step
    # copies its inputs (x, Wqkv, Wo, dout) from pinned host memory and its
    # results (out, LSE, dx, dWqkv, dWo) back.  Two device buffer sets let
    # step k + 1's host->device copies run on a copy stream while step k
    # computes, and step k's device->host copies while step k + 1 computes
    # (a pipelined loader); the timed region opens before the first copy and
    # closes after the last, so every byte of every step crosses inside it.
    e2e = None
    if rank == 0 or world > 1:
        pin = lambda t: t.to("cpu").pin_memory()
        hx, hw, hwo, hd = pin(x), pin(wqkv), pin(wo), pin(dout)
        ho, hl, hdx, hdw, hdwo = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                                  for t in (out, lse, dx, dwqkv, dwo))
        h2d = _bytes(hx, hw, hwo, hd)
        d2h = _bytes(ho, hl, hdx, hdw, hdwo)
        k_e2e = max(3, min(args.steps, 10))
        sets = [(x, wqkv, wo, dout, out, lse, dx, dwqkv, dwo),
                tuple(torch.empty_like(t) for t in (x, wqkv, wo, dout, out, lse, dx, dwqkv, dwo))]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ready = [torch.cuda.Event(), torch.cuda.Event()]    # inputs of buffer set b landed
        done = [torch.cuda.Event(), torch.cuda.Event()]     # compute on buffer set b finished
        free = [torch.cuda.Event(), torch.cuda.Event()]     # buffer set b's results copied out

        def load(b):
            s_in.wait_event(free[b])
            with torch.cuda.stream(s_in):
                for dst, src in zip(sets[b][:4], (hx, hw, hwo, hd)):
                    dst.copy_(src, non_blocking=True)
                ready[b].record(s_in)

        def compute(b):
            bx, bw, bwo, bd, bo, bl, bdx, bdw, bdwo = sets[b]
            stream.wait_event(ready[b])
            layer_step(args.o_mode, bx, bw, bwo, bd, bo, bl, bdx, bdw, bdwo)
            done[b].record(stream)
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                for dst, src in zip((ho, hl, hdx, hdw, hdwo), (bo, bl, bdx, bdw, bdwo)):
                    dst.copy_(src, non_blocking=True)
                free[b].record(s_out)

        def run(n):
            for b in (0, 1):
                free[b].record(s_out)
            load(0)
            for k in range(n):
                if k + 1 < n:
                    load((k + 1) % 2)
                compute(k % 2)
            stream.wait_stream(s_out)

        run(2)  # warm-up of the copy path
        torch.cuda.synchronize(dev)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        run(k_e2e)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a0.elapsed_time(a1) / k_e2e, dev)
        e2e = {"value": world * step_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": k_e2e,
               "note": "pinned host buffers; two device buffer sets, host<->device copies on two copy streams "
                       "overlapping the neighbouring steps' compute; all copies inside the timed region"}
        del hx, hw, hwo, hd, ho, hl, hdx, hdw, hdwo, sets

    # ---- activation offload: the block input x to pinned host memory and
    # back on the library's copy streams, alone and beside one layer step.
    offload = None
    if rank == 0 or world > 1:
        hbuf = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hsrc = x.to("cpu").pin_memory()
        dbuf = torch.empty_like(x)
        nbytes = _bytes(x)

        def timed_copies(fn):
            torch.cuda.synchronize(dev)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            fn()
            upipe.copies_join(stream)
            a1.record(stream)
            torch.cuda.synchronize(dev)
            return a0.elapsed_time(a1)

        timed_copies(lambda: (upipe.offload_async(hbuf, x, stream), upipe.prefetch_async(dbuf, hsrc, stream)))
        off_ms = timed_copies(lambda: upipe.offload_async(hbuf, x, stream))
        pre_ms = timed_copies(lambda: upipe.prefetch_async(dbuf, hsrc, stream))
        both_ms = timed_copies(lambda: step())
        with_ms = timed_copies(lambda: (upipe.offload_async(hbuf, x, stream), upipe.prefetch_async(dbuf, hsrc, stream),
                                        step()))
        offload = {"bytes": nbytes, "offload_ms": off_ms, "prefetch_ms": pre_ms,
                   "offload_gbs": nbytes / off_ms / 1e6, "prefetch_gbs": nbytes / pre_ms / 1e6,
                   "step_ms": both_ms, "step_with_copies_ms": with_ms,
                   "note": "x of the workload to pinned host memory and back over the host link, timed alone; "
                           "then one layer step with an x-sized offload and prefetch in flight beside it"}
        if not torch.equal(dbuf, x) or not torch.equal(hbuf, hsrc):
            raise RuntimeError("offload/prefetch round trip changed the data")
        del hbuf, hsrc, dbuf
        check_status("after the offload measurement")

    # ---- peak activation bytes and throughput against U (measured)
    del ws, o_host
    sweep = None
    if not args.no_u_sweep:
        sweep = u_sweep(w, U_SWEEP.get(args.workload, (H, U)), dev, stream, x, wqkv, wo, dout)
        check_status("after the U sweep")
    alst = None
    if not args.no_alst:
        alst = alst_section(args.workload, w, dev, stream)
        check_status("after the tiled MLP and loss")

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        Ls = min(L, args.cpu_sample_L)
        v, s = cpu_oracle_sample(Ls)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 NumPy oracle, one query head (H=Hkv=1) of causal attention fwd+bwd at L={Ls} "
                         f"(BLAS threads: all {os.cpu_count()} host cores), {s:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, **w, "d": 128, "rope_theta": 500000.0, "causal": True,
                   "o": O_MODE_NOTE[args.o_mode], "flops_per_step": step_flops, "attn_flops_per_step": attn_f,
                   "l2": (f"inputs larger than L2 (x, dout {L * D * 2 / 2**20:.0f} MiB each)" if 2 * L * D * 2 > 129e6
                          else f"inputs fit in L2 (x, dout {L * D * 2 / 2**20:.1f} MiB each; not flushed)"),
                   "parallelism": f"replicas x{world}"},
        "pct_bf16_peak": {"burst": value / world / burst, "sustained": value / world / sustained,
                          "target_of_burst": TARGET_FRAC_OF_BURST,
                          "peaks": f"{burst} burst / {sustained} sustained TFLOP/s ({peak_src})"},
        "attention_only": attention,
        "fwd_bwd": {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                    "fwd_tflops": world * (attn_f * 2.0 / 7.0 + proj_f / 3.0) / (fwd_ms / 1e3) / 1e12,
                    "bwd_tflops": world * (attn_f * 5.0 / 7.0 + proj_f * 2.0 / 3.0) / (bwd_ms / 1e3) / 1e12},
        "hfu": {"value": world * (step_flops + recompute_flops) / (ms_step / 1e3) / 1e12, "unit": "TFLOP/s",
                "note": "hardware flops: the layer flops plus the backward's recompute of QKV"
                        + (" and attention fwd" if args.o_mode == "recompute" else "")},
        "other_o_mode": {"o": O_MODE_NOTE[other_mode], "ms_per_step": other_ms,
                         "value": job_tflops(step_flops, other_ms, world), "steps": n_split},
        "roofline": roofline, "kernels": kernels, "profiled_step_ms": prof_step_ms,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks, "u_sweep": sweep, "offload": offload, "alst": alst,
    }
    print(json.dumps(line), flush=True)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="world size: ranks (one per GPU); without torchrun, N > 1 relaunches under it")
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="upipe", choices=["upipe", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--ref-sample-L", type=int, default=8192)
    ap.add_argument("--cpu-sample-L", type=int, default=32768)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-u-sweep", action="store_true")
    ap.add_argument("--no-alst", action="store_true", help="skip the sequence-tiled MLP and loss measurement")
    ap.add_argument("--o-mode", default="host", choices=["host", "recompute"],
                    help="where the attention output O waits between forward and backward")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        # --gpus drives the world size: one process per GPU under torchrun.
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__),
               *sys.argv[1:]]
        sys.exit(subprocess.call(cmd))
    if env_world is not None and int(env_world) != args.gpus:
        sys.exit(f"--gpus {args.gpus} but WORLD_SIZE={env_world}: they must agree")
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, w, world, rank)
        return
    world, rank, local = dist_setup()
    try:
        run_upipe(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
