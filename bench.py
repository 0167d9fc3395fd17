#!/usr/bin/env python
"""Benchmark: causal linear attention (SLiM chunked form), forward + backward.

One step = slim_attn_fwd + slim_attn_bwd over one synthetic batch of the
workload (default ``l32k``: B=2, H=16, L=32768, d=64, M=256, chunk 128, bf16
I/O, FAVOR+ with block-orthogonal W).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

``--impl reference`` times the fp64 CPU oracle on this machine's host cores
on a bounded sample of the same workload (the reference arm).  Multi-GPU runs
(torchrun) are independent replicas: heads are independent problems, so every
rank runs its own copy of the workload and no data crosses ranks.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal linear-attn fwd+bwd tokens/s on 1 GB300; % of roofline; peak mem vs L"
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def work_per_token_head(wl, dw=False):
    """Algorithmic FLOPs and bytes per (token, head): a multiply-add counts 2,
    the causal C x C block counts its triangle, d' = d + 1 carries the
    normaliser, recomputation is excluded; dw: the backward also forms
    dW = sum of x^T u over the q and k rows (4 d M)."""
    d, M, C = wl.d, wl.M, wl.chunk
    dp = d + 1
    s = 4 if wl.dtype == "fp32" else 2
    feat = 4 * d * M if wl.feature == "favor" else 0
    fwd = feat + M * (C + 1) + dp * (C + 1) + 4 * M * dp + d
    bwd = dp * (C + 1) + 2 * M * (C + 1) + d * (C + 1) + 8 * M * dp + 2 * M * d + feat
    if dw and wl.feature == "favor":
        bwd += 4 * d * M
    return {"fwd_flops": fwd, "bwd_flops": bwd, "fwd_bytes": 4 * d * s, "bwd_bytes": 7 * d * s}


# sources whose digest tags a recorded DRAM-traffic figure (profiles/*.md lines
# "traffic: <workload> <token-heads> <kernel> <bytes> sources=<digest>")
KERNEL_SOURCES = {
    "tc_backward": ("tc_backward.cu", "tc_backward_elu.cu", "tc_common.cuh", "common.cuh"),
    "tc_forward": ("tc_forward.cu", "tc_common.cuh", "common.cuh"),
    "tc_backward_fix": ("tc_correction.cu", "tc_backward_elu.cu", "tc_common.cuh", "common.cuh"),
}


def source_digest(kernel):
    import hashlib
    files = KERNEL_SOURCES.get(kernel)
    if files is None:
        return None
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sub_linear_memory_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, wl_name, token_heads):
    """DRAM bytes per launch from an ncu capture recorded under profiles/,
    scaled to this launch's token-heads (the kernels stream each token-head's
    rows once, so traffic grows in proportion); None when no capture of this
    workload exists or the kernel's sources changed since it was taken."""
    digest = source_digest(kernel)
    pdir = os.path.join(ROOT, "profiles")
    if digest is None or not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith(".md"):
            continue
        with open(os.path.join(pdir, fn)) as fh:
            for ln in fh:
                f = ln.split()
                if len(f) == 6 and f[0] == "traffic:" and f[1] == wl_name and f[3] == kernel \
                        and f[5] == "sources=" + digest:
                    return float(f[4]) * token_heads / float(f[2])
    return None


KERNEL_WORK = {
    # kernel name -> which algorithmic unit one launch of it processes in full
    "gen_forward": "fwd", "tc_forward": "fwd",
    "gen_backward": "bwd", "tc_backward": "bwd",
}


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms (read only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return rank, world, local, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(wl, row_frac=1.0, threads=0):
    """Time the oracle (fwd + bwd) on min(2 * cores, B*H) heads of the
    workload, optionally on the first ``row_frac`` of the rows; returns
    (seconds, heads, rows, cores).  Inputs follow the workload recipe on the
    CPU."""
    import oracle
    from sub_linear_memory_gb300 import inputs

    cores = threads or len(os.sched_getaffinity(0))
    heads = min(2 * cores, wl.B * wl.H)
    rows = max(1, int(wl.L * row_frac))
    small = wl.with_(L=rows)
    q, k, v, dy, w = inputs.make_inputs(small, heads=(1, heads))
    qn, kn, vn, dyn = (t.to(torch.float64).numpy() for t in (q, k, v, dy))
    wn = None if w is None else w.to(torch.float64).numpy()
    t0 = time.perf_counter()
    oracle.recurrence_forward(qn, kn, vn, wn, threads=cores)
    oracle.recurrence_backward(qn, kn, vn, wn, dyn, threads=cores, want_dw=False)
    return time.perf_counter() - t0, heads, rows, cores


def tile_errors(got, ref):
    """Error of every 128-row tile of every head over the RMS tile norm of the
    reference (a whole tensor's norm cannot see one wrong tile): returns the
    worst value and its (b, h, tile)."""
    import numpy as np

    B, H, L, d = ref.shape
    nt, full = (L + 127) // 128, L // 128
    parts = [(got[:, :, :full * 128].reshape(B, H, full, 128 * d), ref[:, :, :full * 128].reshape(B, H, full, 128 * d))]
    if full < nt:
        parts.append((got[:, :, full * 128:].reshape(B, H, 1, -1), ref[:, :, full * 128:].reshape(B, H, 1, -1)))
    num = np.concatenate([np.linalg.norm(g - r, axis=3) for g, r in parts], axis=2)
    den = np.concatenate([np.linalg.norm(r, axis=3) for _, r in parts], axis=2)
    err = num / np.sqrt(np.mean(den ** 2))
    at = np.unravel_index(int(err.argmax()), err.shape)
    return float(err.max()), [int(x) for x in at]


def oracle_baseline_and_parity(wl, binding, want_dw, row_frac=1.0):
    """One pass of the fp64 oracle on the host cores, used twice:
    * timed (forward + backward) as the CPU baseline, on min(2 * cores, B*H)
      heads and the first ``row_frac`` of the rows, scaled to the workload;
    * with every row (row_frac = 1), as the parity check of one library
      fwd + bwd on the same inputs, drawn on the CPU and copied to the GPU,
      outside the timed region.
    Returns (cpu_baseline dict, parity dict or None)."""
    import numpy as np

    import oracle
    from sub_linear_memory_gb300 import inputs

    cores = len(os.sched_getaffinity(0))
    bh = wl.B * wl.H
    heads = min(2 * cores, bh)
    rows = max(1, int(wl.L * row_frac))
    q, k, v, dy, w = inputs.make_inputs(wl)  # CPU draws of the full workload

    def head_rows(t):
        return t.reshape(bh, wl.L, wl.d)[:heads, :rows].unsqueeze(0).to(torch.float64).numpy()

    qn, kn, vn, dyn = (head_rows(t) for t in (q, k, v, dy))
    wn = None if w is None else w.to(torch.float64).numpy()
    check_dw = want_dw and w is not None and rows == wl.L
    t0 = time.perf_counter()
    y_ref = oracle.recurrence_forward(qn, kn, vn, wn, threads=cores)
    t_fwd = time.perf_counter() - t0
    grads = oracle.recurrence_backward(qn, kn, vn, wn, dyn, threads=cores, want_dw=check_dw)
    secs = time.perf_counter() - t0
    base = {"value": tokens_per_s_from_sample(wl, secs, heads, rows, cores), "unit": "tokens/s",
            "fwd_value": tokens_per_s_from_sample(wl, t_fwd, heads, rows, cores),
            "cores": cores, "kind": "oracle",
            "sample": "%d of %d heads x first %d of %d rows, fp64 recurrence fwd+bwd (%.1f s), scaled to the full workload"
                      % (heads, bh, rows, wl.L, secs)}
    if rows != wl.L:
        return base, None
    # the library on the same (CPU-drawn) inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    gq, gk, gv, gdy = (t.to(dev) for t in (q, k, v, dy))
    gw = None if w is None else w.to(dev)
    y = binding.slim_attn_fwd(gq, gk, gv, gw, wl.chunk)
    dq, dk, dv, dw = binding.slim_attn_bwd(gq, gk, gv, gw, gdy, wl.chunk, want_dw=check_dw)
    torch.cuda.synchronize()
    binding.sync_status()
    tol = 1e-4 if wl.dtype == "fp32" else 2e-2
    parity = {"heads": "%d of %d" % (heads, bh), "rows": "all %d" % wl.L, "metric": "relative L2 over the heads, fp64",
              "tol": tol, "worst_tile_metric": "error of one 128-row tile over the RMS tile norm, [b, h, tile]",
              "rel_l2": {}, "worst_tile": {}}
    for name, got, ref in (("Y", y, y_ref), ("dQ", dq, grads[0]), ("dK", dk, grads[1]), ("dV", dv, grads[2])):
        g = head_rows(got.cpu())
        parity["rel_l2"][name] = oracle.rel_l2(g, ref)
        worst, at = tile_errors(g, ref)
        parity["worst_tile"][name] = {"err": worst, "at": [at[1] // wl.H, at[1] % wl.H, at[2]]}
    if check_dw:
        parity["rel_l2"]["dW"] = oracle.rel_l2(dw.cpu().to(torch.float64).numpy(), grads[3])
    parity["pass"] = all(e <= tol for e in parity["rel_l2"].values())
    del gq, gk, gv, gdy, y, dq, dk, dv
    return base, parity


def workload_timings(binding, inputs, peaks, names, steps=20, warmup=3):
    """fwd + bwd and forward-alone times of other workloads, each on its own
    device-drawn inputs, outside the main timed region (CUDA events on the
    current stream; inputs larger than L2 except where noted)."""
    out = {}
    stream = torch.cuda.current_stream()
    for name in names:
        wl = inputs.WORKLOADS[name]
        q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
        y = torch.empty_like(q)
        grads = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q), None)

        def timed(fn, n):
            for _ in range(warmup):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        def step():
            binding.slim_attn_fwd(q, k, v, w, wl.chunk, y=y)
            binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk, out=grads)

        ms = timed(step, steps)
        fwd_ms = timed(lambda: binding.slim_attn_fwd(q, k, v, w, wl.chunk, y=y), steps)
        binding.sync_status()
        work = work_per_token_head(wl)
        th = wl.B * wl.H * wl.L
        # timed regions well under a second: the burst tensor peak applies
        roof = lambda fl, nb: max(fl * th / (peaks["bf16_tflops"] * 1e12), nb * th / (peaks["hbm_gbs"] * 1e9))
        t_step = roof(work["fwd_flops"] + work["bwd_flops"], work["fwd_bytes"] + work["bwd_bytes"])
        t_fwd = roof(work["fwd_flops"], work["fwd_bytes"])
        out[name] = {"B": wl.B, "H": wl.H, "L": wl.L, "d": wl.d, "M": wl.M, "chunk": wl.chunk, "feature": wl.feature,
                     "ms_per_step": ms, "tokens_per_s": wl.B * wl.L / (ms / 1e3),
                     "roofline_ms": t_step * 1e3, "frac": t_step * 1e3 / ms,
                     "fwd_ms": fwd_ms, "fwd_tokens_per_s": wl.B * wl.L / (fwd_ms / 1e3), "fwd_frac": t_fwd * 1e3 / fwd_ms,
                     "steps": steps, "peak": "burst bf16 %.1f TFLOP/s, HBM %.1f GB/s (%s)" % (
                         peaks["bf16_tflops"], peaks["hbm_gbs"], peaks["source"])}
        del q, k, v, dy, w, y, grads
        torch.cuda.empty_cache()
    if "l32k" in inputs.WORKLOADS:
        out["l32k_per_head_w_redraw_dw"] = per_head_redraw_timing(binding, inputs, peaks, steps, warmup)
    return out


def per_head_redraw_timing(binding, inputs, peaks, steps=20, warmup=3):
    """The l32k shape with one FAVOR+ projection per head, redrawn on the device
    every step (slim_attn_draw_orf), and dW per head from the backward."""
    wl = inputs.WORKLOADS["l32k"]
    q, k, v, dy, _ = inputs.make_inputs(wl, device="cuda")
    y = torch.empty_like(q)
    w = torch.empty((wl.H, wl.d, wl.M), dtype=torch.float32, device="cuda")
    dw = torch.empty_like(w)
    grads = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q), dw)
    stream = torch.cuda.current_stream()
    binding.set_option(binding.OPT_W_PER_HEAD, 1)
    try:
        it = [0]

        def step():
            binding.draw_orf(wl.H, wl.d, wl.M, seed=2024, step=it[0], out=w)
            it[0] += 1
            binding.slim_attn_fwd(q, k, v, w, wl.chunk, y=y)
            binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk, out=grads)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        binding.sync_status()
    finally:
        binding.set_option(binding.OPT_W_PER_HEAD, 0)
    ms = e0.elapsed_time(e1) / steps
    work = work_per_token_head(wl, dw=True)
    th = wl.B * wl.H * wl.L
    roof = max((work["fwd_flops"] + work["bwd_flops"]) * th / (peaks["bf16_tflops"] * 1e12),
               (work["fwd_bytes"] + work["bwd_bytes"]) * th / (peaks["hbm_gbs"] * 1e9))
    return {"B": wl.B, "H": wl.H, "L": wl.L, "d": wl.d, "M": wl.M, "chunk": wl.chunk,
            "feature": "FAVOR+, one block-orthogonal W per head redrawn on the device every step, dW per head",
            "ms_per_step": ms, "tokens_per_s": wl.B * wl.L / (ms / 1e3), "roofline_ms": roof * 1e3,
            "frac": roof * 1e3 / ms, "steps": steps}


def streamed_timings(binding, inputs, exps=(20, 21, 22), window=1 << 18, steps=5, warmup=2):
    """fwd + bwd of the 1M workload's head shape with Q, K, V, dY (and Y, dQ,
    dK, dV) kept in pinned host memory and run window by window (stream.py):
    CUDA-event time per step on the current stream (the host<->device copies
    are part of the work; the median of the timed steps), the bytes copied,
    and the peak device memory held against L."""
    from sub_linear_memory_gb300 import stream

    base = inputs.WORKLOADS["l1m"]
    out = {"workload": "l1m head shape (B=1, H=8, d=64, M=64, chunk 256), inputs and outputs in pinned host memory",
           "window": window, "timing": "median of %d steps after %d warm-up" % (steps, warmup),
           "L": [], "ms_per_step": [], "tokens_per_s": [], "peak_device_bytes": [],
           "h2d_bytes_per_step": [], "d2h_bytes_per_step": []}
    for e in exps:
        wl = base.with_(L=1 << e)
        dev_inputs = inputs.make_inputs(wl, device="cuda")
        q, k, v, dy = (t.cpu().pin_memory() for t in dev_inputs[:4])
        w = dev_inputs[4]
        del dev_inputs
        y, dq, dk, dv = (torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4))
        nwin = (wl.L + window - 1) // window
        ckpt = torch.empty((nwin, wl.B, wl.H, wl.d + 1, wl.M), dtype=torch.float32).pin_memory()
        binding.release_workspace()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        before = torch.cuda.memory_allocated()

        def step():
            _, ck = stream.streamed_forward(q, k, v, w, wl.chunk, window, y=y, ckpt=ckpt)
            stream.streamed_backward(q, k, v, dy, w, wl.chunk, ck, out=(dq, dk, dv))

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        # each step timed on its own and the median kept: a step here is
        # mostly host-link copies, which another process on the host can slow
        times = []
        for _ in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            step()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        binding.sync_status()
        ms = sorted(times)[len(times) // 2]
        nbytes = q.numel() * q.element_size()
        out["L"].append(wl.L)
        out["ms_per_step"].append(ms)
        out["tokens_per_s"].append(wl.B * wl.L / (ms / 1e3))
        out["peak_device_bytes"].append(int(torch.cuda.max_memory_allocated() - before))
        out["h2d_bytes_per_step"].append(7 * nbytes)  # q, k, v forward; q, k, v, dy backward
        out["d2h_bytes_per_step"].append(4 * nbytes)  # y; dq, dk, dv
        del q, k, v, dy, w, y, dq, dk, dv, ckpt
        binding.release_workspace()
        torch.cuda.empty_cache()
    return out


LM_CONFIG = {"vocab": 256, "d_model": 256, "heads": 4, "d_ff": 1024, "layers": 3, "M": 64}


def lm_timings(binding, B=2, L=4096, chunks=(64, 256, 1024, 4096), steps=2, warmup=1):
    """One loss + gradient evaluation of a 3-layer Performer language model by
    Algorithm 1 (slim_lm_loss_grad), as the SLiM page measures it (section 4):
    wall-clock time (CUDA events) and peak device memory of the call
    (torch.cuda.max_memory_allocated above what was allocated before it: the
    gradient buffer and the workspace; the 10 MB of parameters come on top)
    against the slice size C, on random byte strings with a randomly
    initialised model.  Boundary states are kept as checkpoints in
    pinned host memory; one line per C also times the recovery by
    subtraction (eq. 19), which needs no checkpoints."""
    import numpy as np
    from sub_linear_memory_gb300 import inputs

    c = LM_CONFIG
    cfg = binding.lm_config(c["vocab"], c["d_model"], c["heads"], c["d_ff"], c["layers"], True, c["M"])
    d = c["d_model"] // c["heads"]
    params = torch.tensor(inputs.lm_init_params(c, 11), dtype=torch.float32, device="cuda")
    fw = binding.draw_orf(c["layers"], d, c["M"], seed=11)  # one fixed projection per layer
    tok = torch.tensor(np.random.default_rng(12).integers(0, c["vocab"], size=(B, L)), dtype=torch.int32,
                       device="cuda")
    out = {"model": "Performer LM: vocab %d, d_model %d, %d heads (d %d), d_ff %d, %d layers, FAVOR+ M %d"
                    % (c["vocab"], c["d_model"], c["heads"], d, c["d_ff"], c["layers"], c["M"]),
           "B": B, "L": L, "data": "random strings over 256 symbols, random initialisation",
           "C": [], "ms_per_step": [], "tokens_per_s": [], "peak_device_bytes": [], "checkpoint_host_bytes": [],
           "ms_per_step_recovered_by_subtraction": []}
    for C in chunks:
        for mode in ("checkpoints", "subtraction"):
            ck = None
            if mode == "checkpoints":
                ck = torch.empty(binding.lm_checkpoint_bytes(cfg, B, L, C) // 4, dtype=torch.float32).pin_memory()
            binding.lm_release_workspace()
            binding.release_workspace()
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            torch.cuda.reset_peak_memory_stats()
            before = torch.cuda.memory_allocated()  # parameters, projections, tokens and earlier buffers
            grads = torch.empty_like(params)
            for _ in range(warmup):
                binding.lm_loss_grad(cfg, params, fw, tok, C, grads=grads, checkpoints=ck)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                loss, _ = binding.lm_loss_grad(cfg, params, fw, tok, C, grads=grads, checkpoints=ck)
            e1.record()
            torch.cuda.synchronize()
            binding.sync_status()
            ms = e0.elapsed_time(e1) / steps
            if mode == "checkpoints":
                out["C"].append(C)
                out["ms_per_step"].append(ms)
                out["tokens_per_s"].append(B * L / (ms / 1e3))
                out["peak_device_bytes"].append(int(torch.cuda.max_memory_allocated() - before))
                out["checkpoint_host_bytes"].append(int(ck.numel() * 4))
                out["loss_per_token"] = float(loss) / (B * (L - 1))
            else:
                out["ms_per_step_recovered_by_subtraction"].append(ms)
    binding.lm_release_workspace()
    del params, fw, tok
    torch.cuda.empty_cache()
    return out


def tokens_per_s_from_sample(wl, secs, heads, rows, cores):
    rounds = math.ceil(wl.B * wl.H / heads)
    full_secs = secs * rounds * (wl.L / rows)
    return wl.B * wl.L / full_secs


def run_reference(args, wl):
    rank, world, _, dist = dist_setup(args.gpus)
    if rank != 0:
        return 0
    row_frac = args.ref_row_frac
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, row_frac)
    times = []
    for _ in range(args.steps):
        secs, heads, rows, cores = cpu_oracle_sample(wl, row_frac)
        times.append(secs)
    secs = sum(times) / len(times)
    value = tokens_per_s_from_sample(wl, secs, heads, rows, cores)
    sample = "%d of %d heads x first %d of %d rows per step, fp64 recurrence fwd+bwd, scaled to the full workload" % (
        heads, wl.B * wl.H, rows, wl.L)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wl.B * wl.L / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(wl, n_gpus):
    io = 4 * wl.B * wl.H * wl.L * wl.d * (4 if wl.dtype == "fp32" else 2)
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "L": wl.L, "d": wl.d, "M": wl.M,
            "chunk": wl.chunk, "feature": "FAVOR+ (block-orthogonal W)" if wl.feature == "favor" and wl.w_kind == "orf"
            else ("FAVOR+ (iid W)" if wl.feature == "favor" else "elu+1"),
            "io_dtype": wl.dtype, "global_batch": wl.B * n_gpus, "seq_len": wl.L,
            "parallelism": "replicas x%d" % n_gpus if n_gpus > 1 else "single GPU",
            "l2": "inputs larger than L2 (%.0f MB of Q,K,V,dY vs 129 MB L2); no flush" % (io / 2**20)
            if io > L2_BYTES else "L2 flushed between steps"}


def memory_sweep(binding, inputs, exps=(16, 18, 20)):
    """Peak device memory of one fwd + bwd on the 1M workload's head shape at
    L = 2^e, from torch.cuda.max_memory_allocated (the workspace is a torch
    allocation), split into the Theta(L) I/O tensors and the rest."""
    base = inputs.WORKLOADS["l1m"]
    out = {"L": [], "peak_bytes": [], "io_bytes": [], "workspace_bytes": [], "non_io_bytes": []}
    for e in exps:
        wl = base.with_(L=1 << e)
        binding.release_workspace()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        before = torch.cuda.memory_allocated()
        q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
        y = binding.slim_attn_fwd(q, k, v, w, wl.chunk)
        dq, dk, dv, _ = binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk)
        torch.cuda.synchronize()
        binding.sync_status()
        peak = torch.cuda.max_memory_allocated() - before
        io = sum(t.numel() * t.element_size() for t in (q, k, v, dy, y, dq, dk, dv))
        ws = max(binding.workspace_bytes(wl.B, wl.H, wl.L, wl.d, wl.M, wl.chunk, b) for b in (0, 1))
        out["L"].append(wl.L)
        out["peak_bytes"].append(int(peak))
        out["io_bytes"].append(int(io))
        out["workspace_bytes"].append(int(ws))
        out["non_io_bytes"].append(int(peak - io))
        del q, k, v, dy, w, y, dq, dk, dv
    binding.release_workspace()
    torch.cuda.empty_cache()
    return out


def recompute_flops_per_token_head(wl, state_passes):
    """FLOPs the kernels spend beyond the algorithmic count, per token-head:
    the backward recomputes the forward of every tile (features, A and num')
    and every segment-state pass recomputes the K-side features and the state
    increments."""
    d, M, C, dp = wl.d, wl.M, wl.chunk, wl.d + 1
    favor = wl.feature == "favor"
    fwd_again = (4 * d * M if favor else 0) + M * (C + 1) + dp * (C + 1) + 4 * M * dp
    state_pass = (2 * d * M if favor else 0) + 2 * M * dp
    return fwd_again + state_passes * state_pass


def ex2_ceiling(binding, sm_mhz, wl, ms_per_step, reps=5):
    """The exponential unit's measured rate (slim_attn_probe_ex2: a kernel of
    nothing but dependent 2^x chains) and the time the step's algorithmic
    exponentials (2M per token-head forward, as many backward) would take at
    that rate: a third ceiling next to the tensor and memory peaks."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    blocks, iters = props.multi_processor_count * 8, 8192
    sink = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    for _ in range(2):
        binding.probe_ex2(blocks, iters, sink)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        binding.probe_ex2(blocks, iters, sink)
    e1.record()
    torch.cuda.synchronize()
    binding.sync_status()
    rate = blocks * 256 * iters * 8 * reps / (e0.elapsed_time(e1) / 1e3)
    exps = (4 * wl.M if wl.feature == "favor" else 0) * wl.B * wl.H * wl.L
    out = {"ex2_per_s": rate, "exps_per_step": exps, "ceiling_ms": exps / rate * 1e3,
           "frac": exps / rate * 1e3 / ms_per_step,
           "note": "informational: algorithmic exponentials (2M per token-head forward, 2M backward) at the "
                   "measured rate of the exponential unit"}
    if sm_mhz:
        out["per_sm_per_clk"] = rate / (props.multi_processor_count * sm_mhz * 1e6)
    return out


def oracle_config_timings(names=("tiny", "l4k", "l1m", "elu16k"), max_rows=4096):
    """The fp64 oracle on the host cores for the other configs, forward and
    forward + backward, each on min(2 * cores, B*H) heads and the first
    min(L, max_rows) rows, scaled to the full workload (heads are independent
    and the recurrence is linear in L)."""
    import oracle
    from sub_linear_memory_gb300 import inputs

    cores = len(os.sched_getaffinity(0))
    out = {}
    for name in names:
        wl = inputs.WORKLOADS[name]
        heads = min(2 * cores, wl.B * wl.H)
        rows = min(wl.L, max_rows)
        q, k, v, dy, w = inputs.make_inputs(wl.with_(L=rows), heads=(1, heads))
        qn, kn, vn, dyn = (t.to(torch.float64).numpy() for t in (q, k, v, dy))
        wn = None if w is None else w.to(torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.recurrence_forward(qn, kn, vn, wn, threads=cores)
        t1 = time.perf_counter()
        oracle.recurrence_backward(qn, kn, vn, wn, dyn, threads=cores, want_dw=False)
        t2 = time.perf_counter()
        out[name] = {"fwd_tokens_per_s": tokens_per_s_from_sample(wl, t1 - t0, heads, rows, cores),
                     "fwd_bwd_tokens_per_s": tokens_per_s_from_sample(wl, t2 - t0, heads, rows, cores),
                     "cores": cores, "sample": "%d of %d heads x first %d of %d rows" % (heads, wl.B * wl.H, rows, wl.L)}
    return out


def run_native(args, wl):
    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    from sub_linear_memory_gb300 import binding, inputs

    peaks = load_peaks()
    # the backward reads the boundary states the forward of the same step left
    # in the workspace (SLIM_OPT_REUSE_STATES) instead of recomputing them
    binding.set_option(binding.OPT_REUSE_STATES, 1 if args.reuse else 0)
    q, k, v, dy, w = inputs.make_inputs(wl, device="cuda")
    y = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    # learnable W: the backward also returns dW (fp32 [d, M])
    dw = torch.empty((wl.d, wl.M), dtype=torch.float32, device=q.device) if (args.dw and w is not None) else None
    out = (dq, dk, dv, dw)

    def step():
        binding.slim_attn_fwd(q, k, v, w, wl.chunk, y=y)
        binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk, out=out)

    for _ in range(args.warmup):
        step()
    binding.sync_status()
    torch.cuda.synchronize()

    # timed region: K steps, barrier + synchronize on both sides, CUDA events
    stream = torch.cuda.current_stream()
    binding.profile_reset()
    binding.profile_enable(True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        host_ms = (time.perf_counter() - h0) * 1e3
    barrier(dist)
    binding.profile_enable(False)
    kernels = binding.profile_read()
    binding.sync_status()
    ev_ms = ev0.elapsed_time(ev1)
    # The events and the host clock bracket the same synchronised region, so
    # the events can only read longer if the GPU's clock moved while it ran;
    # then the host's time stands.
    timer = {"source": "cuda_events", "event_ms": ev_ms, "host_ms": host_ms}
    if ev_ms > 1.02 * host_ms:
        timer["source"] = "host (the GPU clock moved during the timed region)"
    ms = max_over_ranks(host_ms if ev_ms > 1.02 * host_ms else ev_ms, dist)
    ms_per_step = ms / args.steps
    tokens = wl.B * wl.L
    value = world * tokens * args.steps / (ms / 1e3)

    # forward alone (same inputs), for the forward tokens/s figure
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    f0.record(stream)
    for _ in range(args.steps):
        binding.slim_attn_fwd(q, k, v, w, wl.chunk, y=y)
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_host_ms = (time.perf_counter() - h0) * 1e3
    fwd_ms = f0.elapsed_time(f1)
    if fwd_ms > 1.02 * fwd_host_ms:
        timer["forward_alone"] = "host (the GPU clock moved during the loop)"
        fwd_ms = fwd_host_ms
    fwd_ms /= args.steps
    binding.sync_status()  # a device-side error in these launches fails the run

    # end to end through the public API with pinned host buffers
    hq, hk, hv, hdy = (t.cpu().pin_memory() for t in (q, k, v, dy))
    hy, hdq, hdk, hdv = (torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4))
    e2e_steps = max(2, min(args.steps, 10))
    # End to end: every step copies its inputs from pinned host memory and
    # reads its outputs back. Device buffers are double-buffered by step
    # parity so that the host-to-device copies of step i+1 and the
    # device-to-host copies of step i-1 run on their own streams while step i
    # computes.
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ins = [[torch.empty_like(q) for _ in range(4)] for _ in range(2)]
    outs = [[torch.empty_like(q) for _ in range(4)] for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps, e_start=None, e_stop=None):
        if e_start is not None:
            e_start.record(stream)
        h2d_s.wait_stream(stream)
        for i in range(nsteps):
            b = i % 2
            if i >= 2:
                h2d_s.wait_event(ev_done[b])  # step i-2 no longer reads ins[b]
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(ins[b], (hq, hk, hv, hdy)):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(h2d_s)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_read[b])  # step i-2's outputs have left outs[b]
            o = outs[b]
            binding.slim_attn_fwd(ins[b][0], ins[b][1], ins[b][2], w, wl.chunk, y=o[0])
            binding.slim_attn_bwd(ins[b][0], ins[b][1], ins[b][2], w, ins[b][3], wl.chunk, out=(o[1], o[2], o[3], dw))
            ev_done[b].record(stream)
            d2h_s.wait_event(ev_done[b])
            with torch.cuda.stream(d2h_s):
                for dst, src in zip((hy, hdq, hdk, hdv), o):
                    dst.copy_(src, non_blocking=True)
                ev_read[b].record(d2h_s)
        stream.wait_stream(d2h_s)
        if e_stop is not None:
            e_stop.record(stream)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist) / e2e_steps
    binding.sync_status()
    nbytes = q.numel() * q.element_size()

    # roofline of the dominant kernel (largest share of the timed region).
    # A timed region well under a second runs at the burst tensor peak; the
    # sustained figure (a seconds-long loop under the power cap) applies only
    # to longer regions.
    sustained = ms > 1000.0
    tensor_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak_kind = "sustained" if sustained else "burst"
    work = work_per_token_head(wl, dw is not None)
    th = wl.B * wl.H * wl.L
    dom = max(kernels.items(), key=lambda kv: kv[1][1]) if kernels else None
    roofline = None
    if dom is not None:
        name, (launches, total_ms) = dom
        unit = KERNEL_WORK.get(name)
        avg_s = total_ms / launches / 1e3
        if unit is not None:
            flops = work[unit + "_flops"] * th
            nb = work[unit + "_bytes"] * th
            t_tensor = flops / (tensor_peak * 1e12)
            t_hbm = nb / (peaks["hbm_gbs"] * 1e9)
            if t_tensor >= t_hbm:
                roofline = {"bound": "tensor", "achieved": flops / avg_s / 1e12,
                            "peak": tensor_peak, "unit": "TFLOP/s"}
            else:
                roofline = {"bound": "hbm", "achieved": nb / avg_s / 1e9,
                            "peak": peaks["hbm_gbs"], "unit": "GB/s"}
            roofline["frac"] = roofline["achieved"] / roofline["peak"]
            roofline["traffic"] = recorded_traffic(name, wl.name, th)
            roofline["kernel"] = name
            roofline["avg_launch_ms"] = total_ms / launches
            roofline["peak_source"] = "%s (%s bf16: timed region %.0f ms; HBM: copy bandwidth)" % (
                peaks["source"], peak_kind, ms)
    # the whole step against its roofline (max of FLOPs at tensor peak, bytes at HBM)
    step_flops = (work["fwd_flops"] + work["bwd_flops"]) * th
    step_bytes = (work["fwd_bytes"] + work["bwd_bytes"]) * th
    t_roof = max(step_flops / (tensor_peak * 1e12), step_bytes / (peaks["hbm_gbs"] * 1e9))
    fwd_roof = max(work["fwd_flops"] * th / (tensor_peak * 1e12),
                   work["fwd_bytes"] * th / (peaks["hbm_gbs"] * 1e9))

    launches = sum(n for n, _ in kernels.values())
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian Q, K, V, dY; block-orthogonal random W)",
        "config": dict(config_of(wl, world), **({"learnable_w": "dW computed by the backward"} if dw is not None else {}),
                       state_reuse=("the backward reads the forward's boundary states" if args.reuse
                                    else "the backward recomputes the boundary states")),
        "clocks": clocks.summary(),
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": 4 * nbytes, "d2h_bytes_per_step": 4 * nbytes,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "timer": timer,
        "roofline": roofline,
        "step_roofline": {"peak": peak_kind, "roofline_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_per_step,
                          "fwd_roofline_ms": fwd_roof * 1e3, "fwd_ms": fwd_ms,
                          "fwd_frac": fwd_roof * 1e3 / fwd_ms,
                          "fwd_tokens_per_s": world * tokens / (fwd_ms / 1e3)},
        "kernels": {n: {"launches": c, "total_ms": t, "share": t / max(sum(x[1] for x in kernels.values()), 1e-12)}
                    for n, (c, t) in sorted(kernels.items(), key=lambda kv: -kv[1][1])},
    }
    # hardware FLOPs: the algorithmic count plus what the kernels recompute
    passes = kernels.get("tc_segment_state", (0, 0.0))[0] / max(args.steps, 1)
    rec = recompute_flops_per_token_head(wl, passes)
    line["step_roofline"]["hw_flops_per_token_head"] = work["fwd_flops"] + work["bwd_flops"] + rec
    line["step_roofline"]["recompute_flops_per_token_head"] = rec
    line["step_roofline"]["hw_tflops"] = (step_flops + rec * th) / (ms_per_step / 1e3) / 1e12
    if rank == 0:
        line["mufu"] = ex2_ceiling(binding, line["clocks"].get("sm_mhz"), wl, ms_per_step)
    if args.memory and rank == 0:
        del hq, hk, hv, hdy, hy, hdq, hdk, hdv, ins, outs
        line["memory"] = memory_sweep(binding, inputs)
    if rank == 0 and world == 1 and args.stream:
        # sequences kept in host memory, window by window: device memory vs L
        line["stream"] = streamed_timings(binding, inputs)
    if rank == 0 and world == 1 and args.lm:
        # NEXT: the multi-layer model of the SLiM page, time and memory against C
        line["lm"] = lm_timings(binding)
    if rank == 0 and world == 1 and args.workloads:
        # the other configs, each timed outside the main region
        others = [n for n in ("l4k", "l1m", "elu16k", "l32k") if n != wl.name]
        line["workloads"] = workload_timings(binding, inputs, peaks, others)
        # the serving decode step: 128 sequences of the l32k head shape
        dwl = inputs.WORKLOADS["l32k"].with_(B=128)
        d_ms, d_bytes, _ = decode_timing(binding, inputs, dwl, 50, 5)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        line["decode"] = {"B": dwl.B, "H": dwl.H, "d": dwl.d, "M": dwl.M, "ms_per_step": d_ms,
                          "tokens_per_s": dwl.B * 1e3 / d_ms, "bytes_per_step": d_bytes, "achieved_gbs": d_gbs,
                          "frac": d_gbs / peaks["hbm_gbs"], "steps": 50,
                          "note": "one new row for each of 128 sequences x 16 heads against the fp32 state in HBM"}
    if rank == 0 and world == 1 and args.cpu_baseline:
        base, parity = oracle_baseline_and_parity(wl, binding, dw is not None, args.cpu_row_frac)
        line["cpu_baseline"] = base
        line["cpu_baseline_configs"] = oracle_config_timings(
            tuple(n for n in ("tiny", "l4k", "l1m", "elu16k", "l32k") if n != wl.name))
        if parity is not None:
            line["parity"] = parity
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def decode_timing(binding, inputs, wl, steps, warmup, clock_gpu=None):
    """Serving step: one new row for every (sequence, head), against a state
    carried in HBM (fp32 [B][H][d + 1][M]); B sequences of H heads decode one
    token each per step.  The state (2 x 136 MB read and written per step at
    128 x 16 heads, d = 64, M = 256) is larger than L2, so no flush is needed.
    Returns (ms per step, bytes per step, clock summary or None)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    b, h, d, m = wl.B, wl.H, wl.d, wl.M
    dtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    g = torch.Generator(device="cpu").manual_seed(4321)
    nsteps = warmup + steps
    scale = 1.0 if wl.feature == "elu" else d ** -0.25
    qkv = (torch.randn((3, nsteps, b, h, d), generator=g) * torch.tensor([scale, scale, 1.0]).view(3, 1, 1, 1, 1))
    qkv = qkv.to(dev, dtype).contiguous()
    _, _, _, _, w = inputs.make_inputs(wl.with_(B=1, H=1, L=1))
    w = None if w is None else w.to(dev)
    # prompt: a short prefill, so the state holds realistic magnitudes
    kp = (torch.randn((b, h, 256, d), generator=g) * scale).to(dev, dtype)
    vp = torch.randn((b, h, 256, d), generator=g).to(dev, dtype)
    state = binding.slim_attn_state(kp, vp, w, wl.chunk)
    y = torch.empty((b, h, d), dtype=dtype, device=dev)
    del kp, vp
    for i in range(warmup):
        binding.slim_attn_decode(qkv[0, i], qkv[1, i], qkv[2, i], w, state, y)
    binding.sync_status()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clock_gpu) if clock_gpu is not None else None
    if clk is not None:
        clk.__enter__()
    e0.record()
    for i in range(warmup, nsteps):
        binding.slim_attn_decode(qkv[0, i], qkv[1, i], qkv[2, i], w, state, y)
    e1.record()
    torch.cuda.synchronize()
    if clk is not None:
        clk.__exit__(None, None, None)
    binding.sync_status()
    ms = e0.elapsed_time(e1) / steps
    s_io = 2 if dtype == torch.bfloat16 else 4
    nbytes = 2 * b * h * (d + 1) * m * 4 + 4 * b * h * d * s_io + (0 if w is None else d * m * 4)
    del qkv, state, y
    return ms, nbytes, (clk.summary() if clk is not None else None)


def run_decode(args, wl):
    from sub_linear_memory_gb300 import binding, inputs

    torch.cuda.set_device(0)
    ms, nbytes, clocks = decode_timing(binding, inputs, wl, args.steps, args.warmup, clock_gpu=0)
    b, h, d, m = wl.B, wl.H, wl.d, wl.M
    peaks = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {
        "metric": "decode tokens/s (one new row for each of B sequences, all heads)",
        "value": b * 1e3 / ms, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 state, %s I/O" % wl.dtype, "data": "synthetic (seeded Gaussian rows, prefill of 256 rows)",
        "config": {"workload": "decode (%s head shape)" % wl.name, "B": b, "H": h, "d": d, "M": m,
                   "feature": wl.feature, "l2": "state larger than L2, no flush"},
        "clocks": clocks, "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "decode",
                     "bytes_per_step": nbytes},
    }
    print(json.dumps(out))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="l32k")
    ap.add_argument("--heads", default=None,
                    help="BxH: run the workload's recipe with another batch and head count "
                         "(a reduced case for profiling); the default is the workload's own")
    ap.add_argument("--dw", action="store_true",
                    help="learnable W: the backward also computes dW")
    ap.add_argument("--no-reuse", dest="reuse", action="store_false",
                    help="the backward recomputes the boundary states instead of reading the forward's")
    ap.add_argument("--no-memory", dest="memory", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false",
                    help="skip the oracle pass (CPU baseline and parity check)")
    ap.add_argument("--no-lm", dest="lm", action="store_false",
                    help="skip the multi-layer Performer (Algorithm 1) timings")
    ap.add_argument("--no-stream", dest="stream", action="store_false",
                    help="skip the host-resident (streamed window) timings")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the timings of the other workloads")
    ap.add_argument("--cpu-row-frac", type=float, default=1.0,
                    help="fraction of the rows the CPU-baseline sample covers")
    ap.add_argument("--decode", action="store_true",
                    help="time the serving decode step instead (B defaults to 128 sequences)")
    ap.add_argument("--ref-row-frac", type=float, default=0.125,
                    help="fraction of the rows each reference-arm step covers")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "native":
        ap.error("--warmup must be >= 3")
    from sub_linear_memory_gb300 import inputs

    wl = inputs.WORKLOADS[args.workload]
    if args.heads:
        b, h = (int(x) for x in args.heads.lower().split("x"))
        wl = wl.with_(B=b, H=h)
    if args.decode:
        if not args.heads:
            wl = wl.with_(B=128)
        return run_decode(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_native(args, wl)


if __name__ == "__main__":
    sys.exit(main())
