"""fa_fwd_host (host buffers, copies overlapped with the attention in groups of heads) on the
GPU: every head is its own problem, so for any grouping the result equals fa_fwd's on the
device bit for bit; one case is also checked against the fp64 oracle."""
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


CASES = [(2, 3, 700, 128, True), (1, 5, 300, 64, False), (1, 1, 129, 128, False),
         (3, 4, 256, 64, True)]


@pytest.mark.parametrize("B,H,N,d,causal", CASES, ids=lambda x: str(x))
@pytest.mark.parametrize("n_chunks", [0, 1, 2, 64])
def test_host_matches_device_bitwise(B, H, N, d, causal, n_chunks):
    q, k, v = inputs.attn_inputs(B, H, N, d, seed=7100 + N + d + H)
    scale = 1.0 / math.sqrt(d)
    Od, Ld = binding.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    Oh, Lh = binding.fa_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=scale,
                                 causal=causal, n_chunks=n_chunks)
    assert binding.device_status() == 0
    assert torch.equal(Oh, Od.cpu()) and torch.equal(Lh, Ld.cpu())


def test_host_pageable_no_lse_and_side_stream():
    B, H, N, d = 2, 2, 500, 128
    q, k, v = inputs.attn_inputs(B, H, N, d, seed=7200)
    Od, _ = binding.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = torch.zeros(q.shape, dtype=torch.bfloat16)  # pageable
    Oh, Lh = binding.fa_fwd_host(q, k, v, causal=True, out=out, return_lse=False, n_chunks=3,
                                 stream=s)
    assert Lh is None and Oh is out
    assert binding.device_status() == 0
    assert torch.equal(Oh, Od.cpu())


def test_host_against_oracle():
    B, H, N, d = 1, 3, 333, 64
    q, k, v = inputs.attn_inputs(B, H, N, d, seed=7300)
    scale = 1.0 / math.sqrt(d)
    Oh, Lh = binding.fa_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=scale,
                                 causal=False, n_chunks=2)
    Oref, Lref = oracle.attention(q, k, v, scale, False)
    parity.check_attention(Oh.float().numpy(), Lh.numpy(), Oref, Lref, "fa_fwd_host")
    assert np.isfinite(Oh.float().numpy()).all()
