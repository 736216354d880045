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


def run(q, k, v, mask, causal, scale=None, skip=True):
    O, L = binding.fa_fwd_mask(q.cuda(), k.cuda(), v.cuda(), bits(mask), scale=scale,
                               causal=causal, skip_tiles=skip)
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


@pytest.mark.parametrize("skip", [False, True], ids=["all_tiles", "tile_map"])
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,mshape,dens,frows,fkeys", CASES,
                         ids=lambda x: str(x))
def test_mask_parity(B, H, Nq, Nk, d, causal, mshape, dens, frows, fkeys, skip):
    q, k, v = qkv(B, H, Nq, Nk, d, seed=8000 + Nq + Nk + d)
    m = inputs.random_mask(mshape[0], mshape[1], Nq, Nk, dens, seed=8100 + Nq,
                           full_rows=frows, full_keys=fkeys)
    O, L = run(q, k, v, m, causal, skip=skip)
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


@pytest.mark.parametrize("skip", [False, True], ids=["all_tiles", "tile_map"])
def test_structured_masks(skip):
    """A sliding window inside documents and a prefix-LM mask, the shapes such masks take (with
    the tile map, most key tiles of the window mask are skipped)."""
    B, H, N, d = 1, 2, 640, 64
    q, k, v = qkv(B, H, N, N, d, seed=8300)
    win = inputs.window_mask(N, N, window=96, doc_len=200)
    O, L = run(q, k, v, win, False, skip=skip)
    Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), False, win)
    parity.check_attention_allow_empty(O, L, Oref, Lref, "window")
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    plm = ((j < 150) | (j <= i)).astype(np.uint8)[None, None]
    O, L = run(q, k, v, plm, False, skip=skip)
    Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), False, plm)
    parity.check_attention_allow_empty(O, L, Oref, Lref, "prefix LM")


@pytest.mark.parametrize("d", [64, 128])
def test_tile_map_skips_whole_tiles(d):
    """Block-sparse masks where the tile map leaves key tiles, and for one query tile every key
    tile, out: per-head block-diagonal masks with ragged blocks (3 tiles of keys per head
    skipped), a query tile with no allowed key at all (O = 0, LSE = -inf for its rows), masks
    shared over sequences, and causal on top.  Both paths against the oracle, and against each
    other to the rounding of the sums."""
    B, H, Nq, Nk = 2, 3, 520, 700
    q, k, v = qkv(B, H, Nq, Nk, d, seed=8500 + d)
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    m = np.zeros((1, H, Nq, Nk), np.uint8)
    for h in range(H):
        blk = 150 + 40 * h  # ragged blocks that straddle tile edges
        m[0, h] = ((i // blk) == (j // blk)) | (j < 10 * h)
    m[:, :, 256:384] = 0  # query tile 2: nothing allowed
    for causal in (False, True):
        Oref, Lref = oracle.attention_masked(q, k, v, 1.0 / math.sqrt(d), causal, m)
        assert np.isinf(Lref[:, :, 256:384]).all()
        O0, L0 = run(q, k, v, m, causal, skip=False)
        O1, L1 = run(q, k, v, m, causal, skip=True)
        for O, L, what in ((O0, L0, "all tiles"), (O1, L1, "tile map")):
            parity.check_attention_allow_empty(O, L, Oref, Lref, f"block sparse {what} {causal}")
            assert (O[:, :, 256:384] == 0).all() and np.isneginf(L[:, :, 256:384]).all()
        fin = np.isfinite(L0)
        assert np.array_equal(fin, np.isfinite(L1))
        assert np.abs(O0 - O1).max() <= 2 ** -7 and np.abs(L0[fin] - L1[fin]).max() <= 1e-5


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
