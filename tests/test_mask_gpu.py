"""fa_fwd_mask (explicit attention masks) on the GPU through the C ABI, against the fp64 oracle
on the same seeded inputs and masks."""
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


def bits(mask):
    return torch.from_numpy(inputs.pack_mask(mask).view(np.int32)).cuda()


def run(q, k, v, mask, causal, scale=None):
    O, L = binding.fa_fwd_mask(q.cuda(), k.cuda(), v.cuda(), bits(mask), scale=scale,
                               causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return O.float().cpu().numpy(), L.cpu().numpy()


def qkv(B, H, Nq, Nk, d, seed):
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=seed)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=seed + 1)
    return q, k, v


# (B, H, Nq, Nk, d, causal, mask shape (Bm, Hm), density, fully masked rows, keys)
CASES = [
    (1, 2, 256, 256, 64, False, (1, 2), 0.5, 1, 1),
    (2, 2, 300, 500, 128, False, (2, 1), 0.8, 2, 3),   # ragged, per-sequence mask
    (2, 3, 384, 384, 128, True, (1, 1), 0.7, 1, 0),    # one mask for all heads, with causal
    (1, 2, 129, 700, 64, False, (1, 2), 0.05, 0, 0),   # sparse: many empty words
    (2, 2, 200, 200, 64, True, (2, 2), 0.95, 3, 2),
    (1, 1, 5, 1000, 128, False, (1, 1), 0.3, 1, 4),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,mshape,dens,frows,fkeys", CASES,
                         ids=lambda x: str(x))
def test_mask_parity(B, H, Nq, Nk, d, causal, mshape, dens, frows, fkeys):
    q, k, v = qkv(B, H, Nq, Nk, d, seed=8000 + Nq + Nk + d)
    m = inputs.random_mask(mshape[0], mshape[1], Nq, Nk, dens, seed=8100 + Nq,
                           full_rows=frows, full_keys=fkeys)
    O, L = run(q, k, v, m, causal)
    Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), causal, m)
    if frows:
        assert np.isinf(Lref).any()
    parity.check_attention_allow_empty(O, L, Oref, Lref, f"{(B, H, Nq, Nk, d, causal, mshape)}")


def test_all_ones_mask_is_unmasked_attention_bit_for_bit():
    """With every bit set the mask step changes nothing: the outputs equal fa_fwd's exactly."""
    q, k, v = qkv(2, 2, 512, 512, 128, seed=8200)
    O, L = run(q, k, v, np.ones((1, 1, 512, 512), np.uint8), False)
    O2, L2 = binding.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    assert np.array_equal(O, O2.float().cpu().numpy()) and np.array_equal(L, L2.cpu().numpy())


def test_structured_masks():
    """A sliding window inside documents and a prefix-LM mask, the shapes such masks take."""
    B, H, N, d = 1, 2, 640, 64
    q, k, v = qkv(B, H, N, N, d, seed=8300)
    win = inputs.window_mask(N, N, window=96, doc_len=200)
    O, L = run(q, k, v, win, False)
    Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), False, win)
    parity.check_attention_allow_empty(O, L, Oref, Lref, "window")
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    plm = ((j < 150) | (j <= i)).astype(np.uint8)[None, None]
    O, L = run(q, k, v, plm, False)
    Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), False, plm)
    parity.check_attention_allow_empty(O, L, Oref, Lref, "prefix LM")


def test_masked_keys_cannot_matter():
    """Huge keys and values at positions masked for every query change nothing."""
    q, k, v = qkv(1, 2, 256, 384, 128, seed=8400)
    m = inputs.random_mask(1, 2, 256, 384, 0.9, seed=8401)
    m[:, :, :, 200:260] = 0
    O, L = run(q, k, v, m, False)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 200:260] = 20.0
    v2[:, :, 200:260] = -500.0
    O2, L2 = run(q, k2, v2, m, False)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


@pytest.mark.parametrize("name", list(inputs.MASK_WORKLOADS))
def test_mask_workloads_full_size_sampled(name):
    """The bench's mask workloads at full size, on seeded sampled rows."""
    w = inputs.MASK_WORKLOADS[name]
    q, k, v = inputs.attn_inputs(w.B, w.H, w.N, w.d, w.seed)
    m = w.mask()
    O, L = binding.fa_fwd_mask(q.cuda(), k.cuda(), v.cuda(), bits(m), scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    g = torch.Generator().manual_seed(w.seed * 7919 + 31)
    rows = np.concatenate([bh * w.N + np.unique(np.r_[torch.randperm(w.N, generator=g)[:24].numpy(),
                                                     w.N - 1])
                           for bh in range(w.B * w.H)])
    Oref, Lref = oracle.attention_masked(q, k, v, w.scale, False, m, rows=rows)
    Og = O.float().cpu().numpy().reshape(-1, w.d)[rows]
    Lg = L.cpu().numpy().reshape(-1)[rows]
    parity.check_attention_allow_empty(Og, Lg, Oref, Lref, name)
