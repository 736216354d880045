"""fa_fwd_gqa_mask (grouped key/value heads, key lengths, an explicit mask and split keys in one
call) on the GPU through the C ABI, against the fp64 oracle on the same seeded inputs."""
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


# (B, H, H_kv, Nq, Nk, d, causal, mask shape (Bm, Hm), density, kv_lens, n_splits,
#  fully masked rows, fully masked keys)
CASES = [
    (2, 4, 2, 256, 700, 64, False, (2, 4), 0.6, [700, 333], 1, 1, 2),
    (2, 4, 1, 300, 900, 128, True, (1, 1), 0.8, [900, 500], 3, 0, 1),   # MQA, causal, 3 ranges
    (1, 8, 2, 1, 4096, 128, False, (1, 8), 0.5, None, 0, 0, 0),        # one query, auto split
    (2, 2, 2, 129, 1000, 64, True, (2, 1), 0.9, [0, 700], 4, 2, 0),    # an empty sequence
    (1, 4, 4, 200, 200, 128, False, (1, 4), 0.3, None, 2, 1, 3),       # H_kv = H, split
    (1, 6, 3, 384, 384, 64, True, (1, 1), 1.0, [384], 1, 0, 0),        # all-ones mask
]


@pytest.mark.parametrize("skip", [False, True], ids=["all_tiles", "tile_map"])
@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,mshape,dens,lens,splits,frows,fkeys", CASES,
                         ids=lambda x: str(x))
def test_gqa_mask_parity(B, H, Hkv, Nq, Nk, d, causal, mshape, dens, lens, splits, frows,
                         fkeys, skip):
    seed = 8600 + Nq + Nk + d + H
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=seed)
    _, k, v = inputs.attn_inputs(B, Hkv, Nk, d, seed=seed + 1)
    m = inputs.random_mask(mshape[0], mshape[1], Nq, Nk, dens, seed=seed + 2, full_rows=frows,
                           full_keys=fkeys)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    scale = 1.0 / math.sqrt(d)
    O, L = binding.fa_fwd_gqa_mask(q.cuda(), k.cuda(), v.cuda(), bits(m), kv_lens=kl,
                                   n_splits=splits, scale=scale, causal=causal, skip_tiles=skip)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    Oref, Lref = oracle.load().attention_gqa(q, k, v, scale, causal,
                                             kv_lens=np.array(lens, dtype=np.int32)
                                             if lens is not None else None, mask=m)
    parity.check_attention_allow_empty(O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref,
                                       f"gqa_mask {B, H, Hkv, Nq, Nk, d, causal, splits}")


def test_gqa_mask_split_equals_one_pass():
    """The key ranges' partial states merged equal one pass up to rounding ([SS] two-worker
    merge): same inputs, mask and lengths, 1 and 5 ranges."""
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 200, 1500, 128
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=8700)
    _, k, v = inputs.attn_inputs(B, Hkv, Nk, d, seed=8701)
    m = inputs.random_mask(1, H, Nq, Nk, 0.7, seed=8702, full_rows=1, full_keys=1)
    kl = torch.tensor([1500, 901], dtype=torch.int32, device="cuda")
    qd, kd, vd, mb = q.cuda(), k.cuda(), v.cuda(), bits(m)
    O1, L1 = binding.fa_fwd_gqa_mask(qd, kd, vd, mb, kv_lens=kl, n_splits=1)
    O5, L5 = binding.fa_fwd_gqa_mask(qd, kd, vd, mb, kv_lens=kl, n_splits=5)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    parity.check_attention_allow_empty(O5.float().cpu().numpy(), L5.cpu().numpy(),
                                       O1.float().cpu().numpy().astype(np.float64),
                                       L1.cpu().numpy().astype(np.float64), "split vs one pass")
