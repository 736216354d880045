"""fa_fwd_gqa (grouped key/value heads, per-sequence key lengths, optional key split) on the GPU
through the C ABI, against the fp64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
from online_softmax_tiled_attn_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    binding.lib()


def qkv(B, H, H_kv, Nq, Nk, d, seed, qk_std=1.0):
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=seed, qk_std=qk_std)
    _, k, v = inputs.attn_inputs(B, H_kv, Nk, d, seed=seed + 1, qk_std=qk_std,
                                 v_dist="uniform" if qk_std > 1.0 else "normal")
    return q, k, v


def run(q, k, v, kv_lens, causal, n_splits):
    lens = None if kv_lens is None else torch.tensor(kv_lens, dtype=torch.int32).cuda()
    O, L = binding.fa_fwd_gqa(q.cuda(), k.cuda(), v.cuda(), kv_lens=lens, n_splits=n_splits,
                              causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return O.float().cpu().numpy(), L.cpu().numpy()


# (B, H, H_kv, Nq, Nk, d, causal, kv_lens, n_splits)
CASES = [
    (2, 8, 2, 300, 300, 128, True, [300, 130], 1),
    (2, 8, 2, 256, 256, 64, False, [1, 256], 1),
    (3, 4, 1, 200, 500, 128, False, [0, 129, 500], 1),   # a sequence with no key at all
    (2, 4, 4, 129, 129, 64, True, [128, 127], 1),        # one key/value head per query head
    (1, 6, 3, 384, 384, 128, True, None, 1),              # grouped heads, no lengths
    (4, 16, 4, 1, 3000, 128, False, [3000, 1, 2999, 1500], 0),  # decode, library-chosen split
    (2, 8, 2, 64, 1024, 64, True, [1024, 700], 0),
    (2, 4, 2, 5, 900, 64, False, [0, 640], 3),            # explicit split, one empty sequence
    (1, 8, 1, 1000, 1000, 64, True, [1000], 1),           # multi-query: one key/value head
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,d,causal,kv_lens,n_splits", CASES,
                         ids=lambda x: str(x))
def test_gqa_parity(B, H, H_kv, Nq, Nk, d, causal, kv_lens, n_splits):
    q, k, v = qkv(B, H, H_kv, Nq, Nk, d, seed=7000 + Nq + Nk + d + H_kv)
    scale = 1.0 / math.sqrt(d)
    O, L = run(q, k, v, kv_lens, causal, n_splits)
    lens = None if kv_lens is None else np.array(kv_lens, np.int32)
    Oref, Lref = oracle.attention_gqa(q, k, v, scale, causal, kv_lens=lens)
    parity.check_attention_allow_empty(O, L, Oref, Lref, f"{(B, H, H_kv, Nq, Nk, d, causal)}")


def test_gqa_high_logits_ragged_lengths():
    """Logits of sd 9 (the ragged stress workload's distribution) with ragged key lengths."""
    B, H, H_kv, N, d = 3, 8, 2, 700, 128
    q, k, v = qkv(B, H, H_kv, N, N, d, seed=7777, qk_std=3.0)
    lens = [700, 333, 128]
    O, L = run(q, k, v, lens, False, 1)
    Oref, Lref = oracle.attention_gqa(q, k, v, 1.0 / math.sqrt(d), False,
                                      kv_lens=np.array(lens, np.int32))
    parity.check_attention_allow_empty(O, L, Oref, Lref, "high logits, ragged lengths")


def test_gqa_equals_repeated_heads_exactly():
    """Grouped heads read the same key/value tiles as plain attention with the key/value heads
    repeated, in the same order: the outputs agree bit for bit."""
    B, H, H_kv, N, d = 2, 8, 2, 512, 64
    q, k, v = qkv(B, H, H_kv, N, N, d, seed=7100)
    O, L = run(q, k, v, None, True, 1)
    rep = H // H_kv
    kr = k.repeat_interleave(rep, dim=1).contiguous()
    vr = v.repeat_interleave(rep, dim=1).contiguous()
    O2, L2 = binding.fa_fwd(q.cuda(), kr.cuda(), vr.cuda(), causal=True)
    torch.cuda.synchronize()
    assert np.array_equal(O, O2.float().cpu().numpy())
    assert np.array_equal(L, L2.cpu().numpy())


def test_key_lengths_ignore_what_lies_beyond():
    """Whatever sits in K and V past a sequence's length cannot change its output."""
    B, H, H_kv, N, d = 2, 4, 2, 384, 128
    q, k, v = qkv(B, H, H_kv, N, N, d, seed=7200)
    lens = [200, 301]
    O, L = run(q, k, v, lens, False, 1)
    k2, v2 = k.clone(), v.clone()
    for b, n in enumerate(lens):
        k2[b, :, n:] = 20.0
        v2[b, :, n:] = -500.0
    O2, L2 = run(q, k2, v2, lens, False, 1)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def _sample(w, per_head, seed_offset=0):
    g = torch.Generator().manual_seed(int(w.seed) * 7919 + 29 + seed_offset)
    out = []
    for bh in range(w.B * w.H):
        k = min(per_head, w.Nq)
        idx = torch.randperm(w.Nq, generator=g)[:k]
        idx[0] = w.Nq - 1  # the last row sees the most keys
        out.append(torch.unique(idx).to(torch.int64) + bh * w.Nq)
    return torch.cat(out).numpy()


@pytest.mark.parametrize("name", list(inputs.GQA_WORKLOADS))
def test_gqa_workloads_full_size_sampled(name):
    """The grouped-head bench workloads at full size, in the bench's launch configuration
    (the library's split choice), on seeded sampled rows."""
    w = inputs.GQA_WORKLOADS[name]
    q, k, v = inputs.gqa_inputs(w)
    lens = None if w.kv_lens is None else torch.tensor(w.kv_lens, dtype=torch.int32).cuda()
    O, L = binding.fa_fwd_gqa(q.cuda(), k.cuda(), v.cuda(), kv_lens=lens, n_splits=w.n_splits,
                              scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    rows = _sample(w, 24)
    Oref, Lref = oracle.attention_gqa(q, k, v, w.scale, w.causal,
                                      kv_lens=None if w.kv_lens is None
                                      else np.array(w.kv_lens, np.int32), rows=rows)
    Og = O.float().cpu().numpy().reshape(-1, w.d)[rows]
    Lg = L.cpu().numpy().reshape(-1)[rows]
    parity.check_attention_allow_empty(Og, Lg, Oref, Lref, name)
