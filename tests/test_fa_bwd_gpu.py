"""fa_bwd (the attention gradients) on the GPU through the C ABI, against the fp64 oracle on the
same seeded inputs.

The forward's O and LSE come from fa_fwd on the GPU, as in training.  Tolerance (derived from
the arithmetic the header declares): the kernel rounds the shares P and dS to bf16 before the
tensor-core products, forms D_i = dO_i . O_i from the bf16 O, and rounds dQ, dK, dV to bf16.
`rounding_model` is the oracle's definition in fp64 with exactly those roundings added; its
distance from the oracle is the error that arithmetic cannot avoid.  Both errors are measured
relative to the gradient's scale (the root mean square of the oracle's entries of that tensor),
and the kernel must stay within 1.2x the model's rms error plus 5e-4 of the scale, and within
2x the model's max error plus 5e-3 of the scale (the max over millions of entries is an
extreme-value statistic: where the kernel's fp32 intermediates round a share differently from
the model's fp64 ones, the two are different samples of the same rounding), under fixed
ceilings that guard against a model gone wrong itself: max |err| <= 0.3 * rms and
rms(err) <= 7.5e-3 * rms.  (The model alone gives rms(err) ~ 2.4e-3 * rms with N(0, 1) inputs and
~5e-3 * rms with logits of sd 9; its max reaches 0.23 * rms on causal rows whose few shares are
large.  Measured on GB300, the kernel's rms error is at most 1.11x the model's and its max
error at most 1.73x.  An extra error uncorrelated with the rounding passes the rms bound only
below about 0.25 % of the gradient's rms.)
"""
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_tiled_attn_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

BWD_MAX_CEIL = 0.3
BWD_RMS_CEIL = 7.5e-3
BWD_RMS_FACTOR, BWD_RMS_SLACK = 1.2, 5e-4
BWD_MAX_FACTOR, BWD_MAX_SLACK = 2.0, 5e-3


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    binding.lib()


def gpu_grads(q, k, v, do, scale, causal):
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, do))
    O, L = binding.fa_fwd(qc, kc, vc, scale=scale, causal=causal)
    dq, dk, dv = binding.fa_bwd(qc, kc, vc, O, gc, L, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def rounding_model(q, k, v, do, scale, causal):
    """The gradients of the definition in fp64 (plain CPU torch), with the kernel's declared
    roundings to bf16: O, the shares P (for dV), dS, and the three outputs."""
    bf = lambda t: t.to(torch.bfloat16).double()  # noqa: E731
    q, k, v, do = (t.double() for t in (q, k, v, do))
    S = scale * (q @ k.transpose(-1, -2))
    if causal:
        n = S.shape[-1]
        S = S.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    P = torch.softmax(S, dim=-1)
    O = bf(P @ v)
    D = (do * O).sum(-1, keepdim=True)
    dS = bf(P * (do @ v.transpose(-1, -2) - D))
    dV = bf(bf(P).transpose(-1, -2) @ do)
    dK = bf(scale * (dS.transpose(-1, -2) @ q))
    dQ = bf(scale * (dS @ k))
    return [t.numpy() for t in (dQ, dK, dV)]


def _rel(err, scale):
    return err.max() / scale, math.sqrt(float(np.mean(err * err))) / scale


def check_grads(got, ref, model, what):
    stats, bad = [], []
    for name, g, r, m in zip(("dQ", "dK", "dV"), got, ref, model):
        assert g.shape == r.shape, what
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        scale = math.sqrt(float(np.mean(r * r))) if r.size else 0.0
        if scale == 0.0:
            # Every dS is 0 in exact arithmetic (one key per row: dP_i0 = D_i); the kernel's
            # fp32 dP - D leaves a residual of its rounding, bounded as in the single-key test.
            assert np.abs(g).max(initial=0.0) <= 1e-4, f"{what}: {name} should be 0"
            continue
        mx, rms = _rel(np.abs(g - r), scale)
        mmx, mrms = _rel(np.abs(m - r), scale)
        stats.append((name, round(mx, 5), round(rms, 6), round(mmx, 5), round(mrms, 6)))
        if mx > min(BWD_MAX_CEIL, BWD_MAX_FACTOR * mmx + BWD_MAX_SLACK):
            bad.append(f"{name} max|err|/rms = {mx:.3e} (rounding model {mmx:.3e})")
        if rms > min(BWD_RMS_CEIL, BWD_RMS_FACTOR * mrms + BWD_RMS_SLACK):
            bad.append(f"{name} rms(err)/rms = {rms:.3e} (rounding model {mrms:.3e})")
    assert not bad, f"{what}: " + "; ".join(bad) + f"  all: {stats}"
    return stats


# (B, H, N, d, causal)
CASES = [
    (1, 1, 128, 64, False),
    (1, 2, 256, 128, False),
    (1, 2, 256, 128, True),
    (2, 2, 300, 64, True),      # ragged last tile
    (1, 3, 500, 128, False),    # ragged, several key and query tiles
    (2, 1, 129, 128, True),     # one row past a tile
    (1, 2, 640, 64, False),
    (1, 1, 1, 64, False),       # a single key
]


@pytest.mark.parametrize("B,H,N,d,causal", CASES, ids=lambda x: str(x))
def test_bwd_parity(B, H, N, d, causal):
    q, k, v, do = inputs.bwd_inputs(B, H, N, d, seed=9000 + N + d + int(causal))
    scale = 1.0 / math.sqrt(d)
    got = gpu_grads(q, k, v, do, scale, causal)
    ref = oracle.attention_bwd(q, k, v, do, scale, causal)
    model = rounding_model(q, k, v, do, scale, causal)
    print(check_grads(got, ref, model, f"{(B, H, N, d, causal)}"))


def test_bwd_single_key_closed_form():
    """With one key the share is 1, so dS = dO.(V - O) = 0: dQ = dK = 0 (up to the fp32 rounding of dP - D), dV = dO."""
    q, k, v, do = inputs.bwd_inputs(1, 2, 1, 128, seed=9100)
    dq, dk, dv = gpu_grads(q, k, v, do, 1.0 / math.sqrt(128), True)
    assert np.abs(dq).max() < 1e-4 and np.abs(dk).max() < 1e-4
    assert np.array_equal(dv, do.float().numpy().astype(np.float64))


def test_bwd_other_scale_and_large_logits():
    """Scores of sd 9 (concentrated shares) and a non-default scale."""
    B, H, N, d = 1, 2, 384, 64
    q, k, v, do = inputs.bwd_inputs(B, H, N, d, seed=9200)
    q, k = (q.float() * 3.0).to(torch.bfloat16), (k.float() * 3.0).to(torch.bfloat16)
    got = gpu_grads(q, k, v, do, 0.1, False)
    ref = oracle.attention_bwd(q, k, v, do, 0.1, False)
    print(check_grads(got, ref, rounding_model(q, k, v, do, 0.1, False), "large logits"))


def test_bwd_deterministic():
    """Every gradient is summed in a fixed order: a second run repeats the first bit for bit."""
    q, k, v, do = inputs.bwd_inputs(1, 2, 512, 128, seed=9300)
    a = gpu_grads(q, k, v, do, 0.088, True)
    b = gpu_grads(q, k, v, do, 0.088, True)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("name", list(inputs.BWD_WORKLOADS))
def test_bwd_workloads_full_size_sampled(name):
    """The bench's backward workloads at full size, in its launch configuration; the oracle
    checks two whole heads (the first and the last), whose gradients depend on no other head."""
    w = inputs.BWD_WORKLOADS[name]
    q, k, v, do = inputs.bwd_inputs(w.B, w.H, w.N, w.d, w.seed)
    got = gpu_grads(q, k, v, do, w.scale, w.causal)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    sl = lambda t: torch.stack([t[b, h] for b, h in heads])[None]  # noqa: E731
    ref = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), w.scale, w.causal)
    model = rounding_model(sl(q), sl(k), sl(v), sl(do), w.scale, w.causal)
    got = [np.stack([g[b, h] for b, h in heads])[None] for g in got]
    print(check_grads(got, ref, model, name))


def rounding_model_gqa(q, k, v, do, scale, causal, lens):
    """rounding_model with grouped key/value heads and key lengths: each key/value head's
    products over its query heads summed in fp64 (fp32 accumulators in the kernel) before the
    one rounding of dK, dV to bf16; keys at or past a length masked; rows with no key give 0."""
    bf = lambda t: t.to(torch.bfloat16).double()  # noqa: E731
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    q, k, v, do = (t.double() for t in (q, k, v, do))
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    allowed = torch.ones(B, 1, N, N, dtype=torch.bool)
    if lens is not None:
        allowed &= (torch.arange(N)[None, :] < torch.tensor(lens)[:, None])[:, None, None, :]
    if causal:
        allowed &= torch.ones(N, N, dtype=torch.bool).tril()[None, None]
    S = (scale * (q @ kr.transpose(-1, -2))).masked_fill(~allowed, float("-inf"))
    P = torch.nan_to_num(torch.softmax(S, dim=-1), nan=0.0)
    O = bf(P @ vr)
    D = (do * O).sum(-1, keepdim=True)
    dS = bf(P * (do @ vr.transpose(-1, -2) - D))
    dV = bf((bf(P).transpose(-1, -2) @ do).reshape(B, Hkv, g, N, d).sum(2))
    dK = bf(scale * (dS.transpose(-1, -2) @ q).reshape(B, Hkv, g, N, d).sum(2))
    dQ = bf(scale * (dS @ kr))
    return [t.numpy() for t in (dQ, dK, dV)]


# (B, H, H_kv, N, d, causal, key lengths)
GQA_CASES = [
    (2, 4, 2, 256, 64, False, [256, 100]),
    (2, 4, 1, 300, 128, True, [300, 129]),     # one key/value head for four query heads
    (1, 8, 2, 384, 128, False, None),
    (3, 2, 2, 200, 64, True, [0, 200, 57]),   # a sequence with no key; H_kv = H
    (1, 6, 3, 129, 128, False, [1]),          # a single key
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,lens", GQA_CASES, ids=lambda x: str(x))
def test_bwd_gqa_parity(B, H, Hkv, N, d, causal, lens):
    """fa_bwd_gqa after fa_fwd_gqa (grouped heads, key lengths) against the oracle's gradients,
    within the rounding model's error."""
    seed = 9400 + N + d + H
    q, _, _ = inputs.attn_inputs(B, H, N, d, seed=seed)
    _, k, v = inputs.attn_inputs(B, Hkv, N, d, seed=seed + 1)
    do, _, _ = inputs.attn_inputs(B, H, N, d, seed=seed + 2)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, do))
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    O, L = binding.fa_fwd_gqa(qc, kc, vc, kv_lens=kl, scale=scale, causal=causal)
    dq, dk, dv = binding.fa_bwd_gqa(qc, kc, vc, O, gc, L, kv_lens=kl, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    lens_np = np.array(lens, np.int32) if lens is not None else None
    ref = oracle.attention_bwd(q, k, v, do, scale, causal, kv_lens=lens_np)
    model = rounding_model_gqa(q, k, v, do, scale, causal, lens)
    print(check_grads(got, ref, model, f"gqa {(B, H, Hkv, N, d, causal, lens)}"))
    if lens is not None:
        for b, n in enumerate(lens):  # keys past the length: exactly zero
            assert np.all(got[1][b, :, n:] == 0) and np.all(got[2][b, :, n:] == 0)


def test_bwd_gqa_matches_mha_entry_point():
    """With H_kv = H and no key lengths fa_bwd_gqa is fa_bwd, bit for bit."""
    q, k, v, do = inputs.bwd_inputs(1, 2, 300, 128, seed=9500)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, do))
    O, L = binding.fa_fwd(qc, kc, vc, causal=True)
    a = binding.fa_bwd(qc, kc, vc, O, gc, L, causal=True)
    b = binding.fa_bwd_gqa(qc, kc, vc, O, gc, L, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
