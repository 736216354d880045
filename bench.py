"""Benchmark of the attention forward (fa_fwd) and the row softmax (osm_softmax) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--quick] [--profile]

One step = one fa_fwd pass over one batch of the workload (every stage of the tiled
online-softmax attention runs inside that one kernel).  Inputs are seeded synthetic bf16
tensors already resident in device memory; L2 is flushed (a 256 MiB write) between timed
steps and each step's kernel is timed with CUDA events on the launching stream.  The JSON
line also carries an end-to-end figure (pinned host buffers, host->device copies, the C-ABI
call and the device->host copy of O and LSE inside the timed region), the roofline of the
kernel, the clocks seen during the timed region, the fp64 CPU oracle timed on the host cores
over a bounded sample, and (unless --quick) the same measurements for the other workloads.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
(batch, head) problems: weak scaling, no collective on the data path); the slowest rank's
time sets the value.  --impl reference times the fp64 CPU oracle instead, on rank 0 only.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (4·B·H·N²·d, causal halved) and % of GB300 dense BF16 peak"
# The non-causal d = 128, N >= 8192 case: the one the >= 60 % of dense bf16 peak target names.
DEFAULT_WORKLOAD = "dense_b2h32n8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_BF16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20


def peaks_raw():
    """MEASURED_PEAKS.json as written, or {} when it is absent."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.t_start = self.t_stop = None

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [ln.strip().split(", ") for ln in self.out if ln.strip()]
        self.out.close()
        os.unlink(self.out.name)
        return self.summarise(rows)

    @staticmethod
    def summarise(rows):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# distributed plumbing (torchrun); only host logic, no collective on the data path
# ---------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def dist_init(backend):
    import torch.distributed as dist

    rank, _, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is None:
        return
    import torch

    if device is not None and device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# GPU measurements
# ---------------------------------------------------------------------------------------------
def time_fa(w, steps, warmup, device, flush, profile=False):
    """Per-launch device time (ms) of fa_fwd on workload w, L2 flushed between launches."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    q, k, v = inputs.workload_inputs(w)
    qd, kd, vd = q.to(device), k.to(device), v.to(device)
    del q, k, v
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        binding.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
    torch.cuda.synchronize(device)
    if profile:
        for _ in range(steps):
            binding.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
        torch.cuda.synchronize(device)
        return None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        binding.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    st = binding.device_status()
    if st != 0:
        raise RuntimeError(f"fa_fwd reported device status {st}")
    return [a.elapsed_time(b) for a, b in ev]


def time_fa_e2e(w, steps, warmup, device):
    """End to end through the public API: fa_fwd_host on pinned host Q, K, V, which copies groups
    of heads to the device, runs the attention and copies O and LSE back, the copies overlapped
    with the attention; each step's copies both ways are inside the timed region."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    q, k, v = inputs.workload_inputs(w)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    del q, k, v
    shape = (w.B, w.H, w.N, w.d)
    dq = torch.empty(shape, dtype=torch.bfloat16, device=device)
    dk, dv, dO = torch.empty_like(dq), torch.empty_like(dq), torch.empty_like(dq)
    dL = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    hO = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    hL = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(device)
    sp = ctypes.c_void_p(int(stream.cuda_stream))

    def step():
        rc = binding.fa_fwd_host_raw(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hO.data_ptr(),
                                     hL.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     dO.data_ptr(), dL.data_ptr(), w.B, w.H, w.N, w.d, w.scale,
                                     w.causal, 0, sp)
        if rc != binding.FA_OK:
            raise RuntimeError(f"fa_fwd_host: {binding.status_string(rc)}")

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    h2d = 3 * hq.numel() * 2
    d2h = hO.numel() * 2 + hL.numel() * 4
    return ms, h2d, d2h


def time_softmax(sw, steps, warmup, device, flush):
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    x = inputs.softmax_workload_inputs(sw).to(device)
    y = torch.empty_like(x)
    lse = torch.empty((sw.rows,), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        binding.osm_softmax(x, out=y, lse=lse)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        binding.osm_softmax(x, out=y, lse=lse)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    return [a.elapsed_time(b) for a, b in ev]


def time_topk(tw, steps, warmup, device, flush):
    """Per-launch device time (ms) of osm_softmax_topk on a top-k workload."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    x = inputs.softmax_inputs(tw.rows, tw.cols, tw.seed, tw.std, tw.spike).to(device)
    vals = torch.empty((tw.rows, tw.k), dtype=torch.float32, device=device)
    idx = torch.empty((tw.rows, tw.k), dtype=torch.int32, device=device)
    lse = torch.empty((tw.rows,), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        binding.osm_softmax_topk(x, tw.k, values=vals, indices=idx, lse=lse)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        binding.osm_softmax_topk(x, tw.k, values=vals, indices=idx, lse=lse)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    return [a.elapsed_time(b) for a, b in ev]


def time_splitkv(w, steps, warmup, device, flush):
    """Per-launch device time (ms) of fa_fwd_splitkv (attention kernel + combine) on a decode
    workload, workspace allocated once outside the timed region."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    q, k, v = inputs.decode_inputs(w)
    qd, kd, vd = q.to(device), k.to(device), v.to(device)
    del q, k, v
    splits, wo, wl = binding.splitkv_plan(w.B, w.H, w.Nq, w.Nk, w.d, 0)
    ws = (torch.empty(max(wo, 1), dtype=torch.float32, device=device),
          torch.empty(max(wl, 1), dtype=torch.float32, device=device))
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def call():
        binding.fa_fwd_splitkv(qd, kd, vd, n_splits=splits, scale=w.scale, causal=w.causal,
                               out=O, lse=L, workspace=ws)

    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if binding.device_status() != 0:
        raise RuntimeError("fa_fwd_splitkv reported a device status")
    return [a.elapsed_time(b) for a, b in ev], splits


def time_gqa(w, steps, warmup, device, flush):
    """Per-launch device time (ms) of fa_fwd_gqa on a grouped-head workload (the key split and
    its workspace, if any, are set up outside the timed region)."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    q, k, v = inputs.gqa_inputs(w)
    qd, kd, vd = q.to(device), k.to(device), v.to(device)
    del q, k, v
    lens = (torch.tensor(w.kv_lens, dtype=torch.int32, device=device)
            if w.kv_lens is not None else None)
    splits, wo, wl = binding.gqa_plan(w.B, w.H, w.H_kv, w.Nq, w.Nk, w.d, w.n_splits)
    ws = (torch.empty(max(wo, 1), dtype=torch.float32, device=device),
          torch.empty(max(wl, 1), dtype=torch.float32, device=device))
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def call():
        binding.fa_fwd_gqa(qd, kd, vd, kv_lens=lens, n_splits=splits, scale=w.scale,
                           causal=w.causal, out=O, lse=L, workspace=ws)

    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if binding.device_status() != 0:
        raise RuntimeError("fa_fwd_gqa reported a device status")
    return [a.elapsed_time(b) for a, b in ev], splits


def time_mask(w, steps, warmup, device, flush):
    """Per-launch device time (ms) of fa_fwd_mask on a mask workload (mask bits made once)."""
    import numpy as np
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    qd, kd, vd = (t.to(device) for t in inputs.attn_inputs(w.B, w.H, w.N, w.d, w.seed))
    mb = torch.from_numpy(inputs.pack_mask(w.mask()).view(np.int32)).to(device)
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    # the tile map workspace, made once; the call's pre-pass refills it every step
    W = 4 * ((w.N + 127) // 128)
    hs = w.N * W if mb.shape[1] == w.H and w.H > 1 else 0
    bs = mb.shape[1] * w.N * W if mb.shape[0] == w.B and w.B > 1 else 0
    tm = torch.empty(max(1, binding.mask_plan(w.B, w.H, w.N, w.N, bs, hs)), dtype=torch.int32,
                     device=device)

    def call():
        binding.fa_fwd_mask(qd, kd, vd, mb, scale=w.scale, out=O, lse=L, skip_tiles=w.tile_map,
                            tile_map=tm)

    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if binding.device_status() != 0:
        raise RuntimeError("fa_fwd_mask reported a device status")
    return [a.elapsed_time(b) for a, b in ev]


def time_bwd(w, steps, warmup, device, flush):
    """Per-call device time (ms) of fa_bwd (its three launches) on a backward workload; the
    forward's O and LSE and the workspace are made outside the timed region."""
    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    qd, kd, vd, gd = (t.to(device) for t in inputs.bwd_inputs(w.B, w.H, w.N, w.d, w.seed))
    O, L = binding.fa_fwd(qd, kd, vd, scale=w.scale, causal=w.causal)
    ws = torch.empty(qd.numel() // w.d, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def call():
        binding.fa_bwd(qd, kd, vd, O, gd, L, scale=w.scale, causal=w.causal, workspace=ws)

    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if binding.device_status() != 0:
        raise RuntimeError("fa_bwd reported a device status")
    return [a.elapsed_time(b) for a, b in ev]


def roofline_tensor(flops, ms, peaks, kind, traffic=None):
    """Against the burst bf16 peak (each launch is timed alone, between L2 flushes); the
    fraction of the sustained peak is given beside it, because a long run of back-to-back
    launches holds the GPU at its power cap as the sustained GEMM loop does."""
    achieved = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_kind": f"burst bf16, {kind}",
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
            "frac_of_nominal_2250": round(achieved / NOMINAL_BF16_TFLOPS, 4)}


def exp_rate(w, ms, peaks_raw, sms=152):
    """The softmax's exponentials per second (one per allowed (query, key) pair: B*H*N^2,
    halved when causal) against the MUFU's ex2 rate, 32 per clock per SM at the measured
    maximum SM clock."""
    n = w.B * w.H * w.N * w.N / (2 if w.causal else 1)
    rate = n / (ms * 1e-3)
    mufu = 32 * sms * float(peaks_raw.get("sm_max_mhz", 2070.0)) * 1e6
    return {"gexp_per_s": round(rate / 1e9, 1), "frac_of_mufu": round(rate / mufu, 4),
            "mufu_gexp_per_s": round(mufu / 1e9, 1)}


def roofline_hbm(nbytes, ms, peaks, kind, traffic=None):
    achieved = nbytes / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_kind": f"copy bandwidth, {kind}"}


# Traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu captures
# summarised under profiles/, one per workload.  Workloads without a capture report None.
NCU_TRAFFIC_BYTES = {
    "mha_b4h16n2048d64": 50398208 + 48640,
    "dense_b2h32n8192": 402727424 + 116288256,
    "causal_b2h32n8192": 582513920 + 119392512,
    "causal_b1h8n32768": 870508800 + 50342912,
    "ragged_b1h16n4000": 49220608 + 384768,
    "decode_b8h32q1k32768d128": 4295275776 + 3711744,
    "gqa_causal_b2h32kv8n8192d128": 363324416 + 102152448,
    "gqa_ragged_b4h32kv8n4096d128": 172562944 + 91484928,
    "gqa_decode_b8h32kv8q1k32768d128": 1073982208 + 5190400,
    "mask_prefixlm_b2h16n4096d128": 102078208 + 13319936,
    "mask_random_b2h16n4096d128": 154048000 + 18532352,
    "mask_window_b2h16n8192d128": 203418112 + 46082816,
    "softmax_65536x4000": 1048660992 + 998156288,
    "softmax_topk_65536x4000_k8": 1048771072 + 6897152,
    "softmax_topk_512x131072_k32": 268552704 + 3390464,
    "softmax_topk_512x131072_k100": 268739840 + 3975680,
    "bwd_b4h16n2048d64": 170481920 + 12257024,
    "bwd_b2h16n8192d128": 675801856 + 156787968,
    "bwd_causal_b2h16n8192d128": 903689728 + 151711744,
}
# The backward workloads: the sum over the call's three kernels (bwd_prep, bwd_kv, bwd_q).


# ---------------------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores, over a bounded sample
# ---------------------------------------------------------------------------------------------
def oracle_rate(w, budget_s=12.0, max_rows=None, seed_offset=0):
    """TFLOP/s of the fp64 oracle on sampled query rows of workload w (about budget_s)."""
    import numpy as np

    import oracle
    from online_softmax_tiled_attn_gb300 import inputs

    q, k, v = inputs.workload_inputs(w)
    total_rows = w.B * w.H * w.N
    g = np.random.default_rng(1234 + seed_offset)

    def row_flops(rows):
        i = rows % w.N
        keys = (i + 1) if w.causal else np.full_like(i, w.N)
        return float(np.sum(4.0 * keys * w.d))

    # calibrate on a small sample, then size the measured sample to the budget
    cal = g.choice(total_rows, size=min(256, total_rows), replace=False)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=cal)
    dt = time.perf_counter() - t0
    per_row = max(dt / len(cal), 1e-7)
    n = int(min(total_rows, max(256, budget_s / per_row)))
    if max_rows:
        n = min(n, max_rows)
    rows = np.sort(g.choice(total_rows, size=n, replace=False))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    dt = time.perf_counter() - t0
    return row_flops(rows) / dt / 1e12, n, total_rows, dt


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, on this workload."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    from online_softmax_tiled_attn_gb300 import inputs

    w = inputs.ATTN_WORKLOADS[args.workload]
    cores = oracle.host_threads()
    budget = max(1.0, min(8.0, 90.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rate(w, budget_s=budget / 4, seed_offset=i)
    vals, secs, rows_done = [], 0.0, 0
    for i in range(args.steps):
        r, n, total, dt = oracle_rate(w, budget_s=budget, seed_offset=100 + i)
        vals.append(r)
        secs += dt
        rows_done += n
    value = statistics.mean(vals)
    sample = (f"{rows_done // max(1, args.steps)} seeded random query rows of {total} per step "
              f"(about {budget:.0f} s of fp64 work per step), all {cores} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, flushed=False),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, flushed=True):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
            "causal": w.causal, "scale": "1/sqrt(d)",
            "inputs": f"bf16 seed {w.seed}, Q,K ~ N(0, sd {w.qk_std}), V "
                      + ("~ N(0,1)" if w.v_dist == "normal" else "~ U(-1,1)"),
            "l2": "flushed between timed steps (256 MiB write)" if flushed else "n/a (CPU)"}


# ---------------------------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--quick", action="store_true", help="skip the other workloads")
    ap.add_argument("--profile", action="store_true",
                    help="launch only (no timing, no flush, no oracle): for ncu captures")
    ap.add_argument("--softmax", action="store_true",
                    help="with --profile: launch osm_softmax instead of fa_fwd")
    ap.add_argument("--decode", action="store_true",
                    help="with --profile: launch fa_fwd_splitkv on the decode workload")
    ap.add_argument("--gqa", default=None,
                    help="with --profile: launch fa_fwd_gqa on this grouped-head workload")
    ap.add_argument("--mask", default=None,
                    help="with --profile: launch fa_fwd_mask on this mask workload")
    ap.add_argument("--bwd", default=None,
                    help="with --profile: launch fa_bwd on this backward workload")
    ap.add_argument("--topk", default=None,
                    help="with --profile: launch osm_softmax_topk on this top-k workload")
    args = ap.parse_args(argv)
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        return run_reference(args)

    import torch

    from online_softmax_tiled_attn_gb300 import binding, inputs

    rank, local, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = dist_init("nccl")
    binding.lib()
    w = inputs.ATTN_WORKLOADS[args.workload]

    if args.profile:
        if args.mask:
            time_mask(inputs.MASK_WORKLOADS[args.mask], args.steps, args.warmup, device, None)
        elif args.bwd:
            time_bwd(inputs.BWD_WORKLOADS[args.bwd], args.steps, args.warmup, device, None)
        elif args.topk:
            time_topk(inputs.TOPK_WORKLOADS[args.topk], args.steps, args.warmup, device, None)
        elif args.gqa:
            time_gqa(inputs.GQA_WORKLOADS[args.gqa], args.steps, args.warmup, device, None)
        elif args.decode:
            dw = next(iter(inputs.DECODE_WORKLOADS.values()))
            time_splitkv(dw, args.steps, args.warmup, device, None)
        elif args.softmax:
            sw = inputs.SOFTMAX_WORKLOADS["softmax_65536x4000"]
            x = inputs.softmax_workload_inputs(sw).to(device)
            for _ in range(args.warmup + args.steps):
                binding.osm_softmax(x)
            torch.cuda.synchronize()
        else:
            time_fa(w, args.steps, args.warmup, device, None, profile=True)
        return 0

    peaks, peaks_kind = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit()
                          else local)
    clocks.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    per_step = time_fa(w, args.steps, args.warmup, device, flush)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    wall = time.perf_counter() - t0
    clk = clocks.stop()

    ms_local = sum(per_step) / len(per_step)
    ms = max_over_ranks(ms_local, dist, device)
    value = world * w.flops / (ms * 1e-3) / 1e12
    e2e_ms, h2d, d2h = time_fa_e2e(w, max(5, args.steps // 10), 3, device)
    e2e_ms = max_over_ranks(e2e_ms, dist, device)
    e2e_value = world * w.flops / (e2e_ms * 1e-3) / 1e12

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w),
        "frac_of_nominal_bf16_2250": round(value / world / NOMINAL_BF16_TFLOPS, 4),
        "roofline": roofline_tensor(w.flops, ms, peaks, peaks_kind,
                                    NCU_TRAFFIC_BYTES.get(w.name)),
        "exp_rate": exp_rate(w, ms, peaks_raw()),
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "clocks": clk,
        "gpu_launches": args.steps,
        "timed_region_wall_s": round(wall, 3),
    }

    if not args.quick:
        other = {}
        for name in [n for n in inputs.ATTN_WORKLOADS if n not in (w.name, "small_b1h1n256d64")]:
            ow = inputs.ATTN_WORKLOADS[name]
            t = time_fa(ow, 20, 3, device, flush)
            oms = max_over_ranks(sum(t) / len(t), dist, device)
            other[name] = {"TFLOP/s": round(world * ow.flops / (oms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(oms, 4),
                           "roofline": roofline_tensor(ow.flops, oms, peaks, peaks_kind,
                                                       NCU_TRAFFIC_BYTES.get(name)),
                           "exp_rate": exp_rate(ow, oms, peaks_raw())}
            torch.cuda.empty_cache()
        for name, dw in inputs.DECODE_WORKLOADS.items():
            t, splits = time_splitkv(dw, 20, 3, device, flush)
            dms = max_over_ranks(sum(t) / len(t), dist, device)
            other[name] = {"GB/s": round(world * dw.hbm_bytes / (dms * 1e-3) / 1e9, 1),
                           "TFLOP/s": round(world * dw.flops / (dms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(dms, 4), "n_splits": splits,
                           "roofline": roofline_hbm(dw.hbm_bytes, dms, peaks, peaks_kind,
                                                    NCU_TRAFFIC_BYTES.get(name))}
            torch.cuda.empty_cache()
        for name, gw in inputs.GQA_WORKLOADS.items():
            t, splits = time_gqa(gw, 20, 3, device, flush)
            gms = max_over_ranks(sum(t) / len(t), dist, device)
            entry = {"TFLOP/s": round(world * gw.flops / (gms * 1e-3) / 1e12, 2),
                     "GB/s": round(world * gw.hbm_bytes / (gms * 1e-3) / 1e9, 1),
                     "ms_per_step": round(gms, 4), "n_splits": splits}
            # One query per head is HBM-bound; longer query blocks are tensor-bound.
            entry["roofline"] = (roofline_hbm(gw.hbm_bytes, gms, peaks, peaks_kind,
                                              NCU_TRAFFIC_BYTES.get(name)) if gw.Nq == 1 else
                                 roofline_tensor(gw.flops, gms, peaks, peaks_kind,
                                                 NCU_TRAFFIC_BYTES.get(name)))
            other[name] = entry
            torch.cuda.empty_cache()
        sw = inputs.SOFTMAX_WORKLOADS["softmax_65536x4000"]
        t = time_softmax(sw, 20, 3, device, flush)
        sms = max_over_ranks(sum(t) / len(t), dist, device)
        other[sw.name] = {"GB/s": round(world * sw.hbm_bytes / (sms * 1e-3) / 1e9, 1),
                          "ms_per_step": round(sms, 4),
                          "roofline": roofline_hbm(sw.hbm_bytes, sms, peaks, peaks_kind,
                                                   NCU_TRAFFIC_BYTES.get(sw.name))}
        for name, tw in inputs.TOPK_WORKLOADS.items():
            t = time_topk(tw, 20, 3, device, flush)
            tms = max_over_ranks(sum(t) / len(t), dist, device)
            other[name] = {"GB/s": round(world * tw.hbm_bytes / (tms * 1e-3) / 1e9, 1),
                           "ms_per_step": round(tms, 4),
                           "roofline": roofline_hbm(tw.hbm_bytes, tms, peaks, peaks_kind,
                                                    NCU_TRAFFIC_BYTES.get(name))}
            torch.cuda.empty_cache()
        for name, mw in inputs.MASK_WORKLOADS.items():
            t = time_mask(mw, 20, 3, device, flush)
            mms = max_over_ranks(sum(t) / len(t), dist, device)
            other[name] = {"TFLOP/s": round(world * mw.flops / (mms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(mms, 4), "tile_map": mw.tile_map,
                           "roofline": roofline_tensor(mw.flops, mms, peaks, peaks_kind,
                                                       NCU_TRAFFIC_BYTES.get(name))}
            torch.cuda.empty_cache()
        for name, bw in inputs.BWD_WORKLOADS.items():
            t = time_bwd(bw, 20, 3, device, flush)
            bms = max_over_ranks(sum(t) / len(t), dist, device)
            other[name] = {"TFLOP/s": round(world * bw.flops / (bms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(bms, 4),
                           "roofline": roofline_tensor(bw.flops, bms, peaks, peaks_kind,
                                                       NCU_TRAFFIC_BYTES.get(name))}
            torch.cuda.empty_cache()
        result["other_workloads"] = other

    if rank == 0:
        import oracle

        rate, n, total, dt = oracle_rate(w, budget_s=12.0)
        result["cpu_baseline"] = {
            "value": round(rate, 6), "unit": "TFLOP/s", "cores": oracle.host_threads(),
            "kind": "oracle",
            "sample": f"{n} seeded random query rows of {total} ({dt:.1f} s of fp64 work)"}
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
