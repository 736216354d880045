"""fa_fwd_splitkv (keys cut into ranges, partial states merged) on the GPU against the fp64
oracle's attention of Nq queries against Nk keys."""
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


def qkv(B, H, Nq, Nk, d, seed):
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=seed)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=seed + 1)
    return q, k, v


def run(q, k, v, causal, n_splits):
    O, L = binding.fa_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), n_splits=n_splits,
                                  causal=causal)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return O.float().cpu().numpy(), L.cpu().numpy()


CASES = [
    (2, 4, 1, 4000, 128, False, 8),
    (2, 4, 1, 4000, 128, True, 8),
    (1, 2, 1, 4096, 64, False, 0),
    (2, 2, 300, 2000, 128, True, 3),
    (1, 1, 128, 128, 64, False, 1),
    (1, 2, 3, 1000, 128, True, 4),
    (1, 1, 200, 100, 64, True, 2),   # more queries than keys: the first 100 rows see no key
    (1, 3, 17, 777, 64, False, 0),
    (3, 1, 1, 129, 128, False, 2),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits", CASES, ids=lambda x: str(x))
def test_splitkv_parity(B, H, Nq, Nk, d, causal, n_splits):
    q, k, v = qkv(B, H, Nq, Nk, d, seed=5000 + Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    O, L = run(q, k, v, causal, n_splits)
    Oref, Lref = oracle.attention_qk(q, k, v, scale, causal)
    parity.check_attention_allow_empty(O, L, Oref, Lref, f"{(B, H, Nq, Nk, d, causal, n_splits)}")


def test_splitkv_explicit_empty_ranges():
    """More ranges than key tiles: the ranges past the keys are empty and must weigh nothing."""
    B, H, Nq, Nk, d = 1, 2, 5, 200, 128
    q, k, v = qkv(B, H, Nq, Nk, d, seed=71)
    n = 7
    rows = B * H * Nq
    ws_o = torch.full((n * rows * d,), float("nan"), device="cuda")
    ws_l = torch.full((n * rows,), float("nan"), device="cuda")
    O = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    L = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rc = binding.fa_fwd_splitkv_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(),
                                    L.data_ptr(), B, H, Nq, Nk, d, 1 / math.sqrt(d), 0, n,
                                    ws_o.data_ptr(), ws_l.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == binding.FA_OK
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.isneginf(ws_l.view(n, rows)[2:]).all()  # ranges 2..6 hold no key
    Oref, Lref = oracle.attention_qk(q, k, v, 1 / math.sqrt(d), False)
    parity.check_attention(O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref)


def test_splitkv_no_keys_and_one_split_equals_fa_fwd():
    q = torch.randn(1, 2, 9, 64).to(torch.bfloat16).cuda()
    e = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    O, L = binding.fa_fwd_splitkv(q, e, e)
    torch.cuda.synchronize()
    assert torch.all(O == 0) and torch.isneginf(L).all()
    q, k, v = inputs.attn_inputs(2, 3, 333, 128, seed=72)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        O1, L1 = binding.fa_fwd(qd, kd, vd, causal=causal)
        O2, L2 = binding.fa_fwd_splitkv(qd, kd, vd, n_splits=1, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_splitkv_plan():
    s, wo, wl = binding.splitkv_plan(8, 32, 1, 32768, 128, 0)
    assert 1 <= s <= 64 and wo == s * 8 * 32 * 128 and wl == s * 8 * 32
    s, wo, wl = binding.splitkv_plan(1, 1, 1, 300, 64, 100)
    assert s == 3  # clamped to the number of 128-key tiles
    s, wo, wl = binding.splitkv_plan(4, 16, 4096, 4096, 64, 1)
    assert s == 1 and wo == 0 and wl == 0
    assert binding.splitkv_plan(1, 1, 1, 0, 64, 0)[0] == 0


@pytest.mark.parametrize("name", list(inputs.DECODE_WORKLOADS))
def test_splitkv_full_size(name):
    w = inputs.DECODE_WORKLOADS[name]
    q, k, v = inputs.decode_inputs(w)
    O, L = run(q, k, v, w.causal, 0)
    Oref, Lref = oracle.attention_qk(q, k, v, w.scale, w.causal)
    parity.check_attention(O, L, Oref, Lref, name)
