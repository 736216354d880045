"""fa_fwd_splitkv_noalloc: the split-key attention for callers that cannot allocate device
memory during a call (a plugin or custom-operator hook whose framework forbids allocation
there, a latency-critical decode loop).  Its partial states live in the library's fixed scratch
array instead of a caller workspace.  Checked through the C ABI against fa_fwd_splitkv with a
workspace, on two calls in a row.  Before each checked call another call with other inputs and
a larger shape fills most of the array with its own partial states, so a (range, row) entry
that the checked call failed to write would be read stale and show up as a mismatch."""
import math

import pytest
import torch

import parity
from online_softmax_tiled_attn_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CASES = [
    (8, 32, 1, 8192, 128, False, 0),
    (1, 2, 3, 1000, 64, True, 4),
    (2, 4, 130, 2048, 128, False, 3),
]


# B1 H16, 128 queries against 8192 keys, d = 128, 15 ranges requested (13 ranges of 5 key
# tiles): 13 * 2048 * 129 = 3.4 Mi floats, 82 % of the 4 Mi-float array.
FILL = (1, 16, 128, 8192, 128, 15)


def _fill_scratch_with_another_call(seed, stream):
    B, H, Nq, Nk, d, n_splits = FILL
    splits, wo, wl = binding.splitkv_plan(B, H, Nq, Nk, d, n_splits)
    assert splits * B * H * Nq * (d + 1) == wo + wl <= 4 << 20
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=7100 + seed, qk_std=2.0)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=7200 + seed, qk_std=2.0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    rc = binding.fa_fwd_splitkv_noalloc_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                            o.data_ptr(), None, B, H, Nq, Nk, d, 0.1, False,
                                            n_splits, stream)
    assert rc == binding.FA_OK, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.device_status() == 0


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits", CASES, ids=lambda x: str(x))
def test_noalloc_matches_workspace_entry_point_twice(B, H, Nq, Nk, d, causal, n_splits):
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=900 + Nk)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=901 + Nk)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(d)
    ref_o, ref_l = binding.fa_fwd_splitkv(qd, kd, vd, n_splits=n_splits, scale=scale,
                                          causal=causal)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        _fill_scratch_with_another_call(seed=call, stream=stream)
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), device="cuda")
        rc = binding.fa_fwd_splitkv_noalloc_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                                o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                                                scale, causal, n_splits, stream)
        assert rc == binding.FA_OK, binding.status_string(rc)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        parity.check_attention(o.float().cpu().numpy(), lse.cpu().numpy(),
                               ref_o.float().cpu().numpy().astype("float64"),
                               ref_l.cpu().numpy().astype("float64"), f"call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 64 ranges x 8192 rows x 129 floats > 4 Mi floats: refused before any launch
    q = torch.zeros(1, 1, 8192, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 8192 * 64, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 3.0)
    rc = binding.fa_fwd_splitkv_noalloc_raw(q.data_ptr(), k.data_ptr(), k.data_ptr(),
                                            o.data_ptr(), None, 1, 1, 8192, 8192 * 64, 128,
                                            0.1, False, 64, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in binding.status_string(rc)
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)
