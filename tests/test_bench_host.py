"""Host-side logic of bench.py, on the CPU: clock-sample parsing, the max-over-ranks timing
with two gloo ranks, and the bounded oracle sample of the CPU baseline."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def test_clock_summary_flags_throttle_reasons():
    rows = [
        ["0", "1965", "2070", "900.1", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["0", "1890", "2070", "1350.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "1500", "2070", "1390.0", "0x8", "Active", "Not Active", "Not Active", "Active"],
        ["garbage"],
    ]
    s = bench.ClockSampler.summarise(rows)
    assert s["samples"] == 3 and s["sm_mhz"] == 1890 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler.summarise([])["sm_mhz"] is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.dist_init("gloo")
    got = bench.max_over_ranks(1.5 + rank, dist)
    bench.barrier(dist)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_single_process_has_no_collective():
    assert bench.max_over_ranks(3.0, None) == 3.0


def test_oracle_rate_is_bounded_and_positive():
    from online_softmax_tiled_attn_gb300 import inputs

    w = inputs.ATTN_WORKLOADS["small_b1h1n256d64"]
    rate, n, total, dt = bench.oracle_rate(w, budget_s=0.2)
    assert rate > 0 and 1 <= n <= total == 256 and dt < 10


def test_workload_flops_match_the_metric_definition():
    from online_softmax_tiled_attn_gb300 import inputs

    w = inputs.ATTN_WORKLOADS["mha_b4h16n2048d64"]
    assert w.flops == 4 * 4 * 16 * 2048 ** 2 * 64
    c = inputs.ATTN_WORKLOADS["causal_b2h32n8192"]
    assert c.flops == 4 * 2 * 32 * 8192 ** 2 * 128 / 2


def test_mask_workload_flops_count_the_allowed_pairs():
    """4 d FLOP per allowed (query, key) pair over every head, against the closed forms of the
    pair counts: prefix-LM row i sees max(prefix, i + 1) keys, a causal window w sees
    min(i + 1, w).  (The random mask's count is its own; making it here takes a minute.)"""
    from online_softmax_tiled_attn_gb300 import inputs

    W = inputs.MASK_WORKLOADS
    p = W["mask_prefixlm_b2h16n4096d128"]
    pairs = sum(max(p.prefix, i + 1) for i in range(p.N))
    assert pairs == p.prefix * p.prefix + sum(range(p.prefix + 1, p.N + 1))
    assert p.flops == 4 * p.d * pairs * p.B * p.H
    w = W["mask_window_b2h16n8192d128"]
    pairs = w.window * (w.window + 1) // 2 + (w.N - w.window) * w.window
    assert w.flops == 4 * w.d * pairs * w.B * w.H
    assert w.tile_map and p.tile_map and not W["mask_random_b2h16n4096d128"].tile_map


def test_ragged_stress_workload_logit_range():
    """The overflow/ragged stress workload draws Q, K with sd 3, so at scale 1/sqrt(128) its
    scaled logits have sd 3 * 3 * sqrt(128) / sqrt(128) = 9; over its 16 x 4000 x 4000 scores
    the largest magnitude observed is about 60 (recorded with the inputs' recipe)."""
    import torch

    from online_softmax_tiled_attn_gb300 import inputs

    w = inputs.ATTN_WORKLOADS["ragged_b1h16n4000"]
    q, k, _ = inputs.workload_inputs(w)
    mx, var = 0.0, 0.0
    for h in range(w.H):
        s = (q[0, h].float() @ k[0, h].float().T) * w.scale
        mx = max(mx, s.abs().max().item())
        var += s.pow(2).mean().item() / w.H
    assert abs(var ** 0.5 - 9.0) < 0.1
    assert 55.0 < mx < 65.0


def test_exp_rate_counts_the_allowed_pairs():
    from online_softmax_tiled_attn_gb300 import inputs

    d = bench.exp_rate(inputs.ATTN_WORKLOADS["dense_b2h32n8192"], 1.0,
                       {"sm_max_mhz": 2000.0})
    assert d["gexp_per_s"] == round(2 * 32 * 8192 ** 2 / 1e-3 / 1e9, 1)
    assert abs(d["frac_of_mufu"] - 2 * 32 * 8192 ** 2 / 1e-3 / (32 * 152 * 2000e6)) < 1e-4
    c = bench.exp_rate(inputs.ATTN_WORKLOADS["causal_b2h32n8192"], 1.0, {"sm_max_mhz": 2000.0})
    assert c["gexp_per_s"] == round(2 * 32 * 8192 ** 2 / 2 / 1e-3 / 1e9, 1)
