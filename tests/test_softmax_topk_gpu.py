"""osm_softmax_topk on the GPU through the C ABI against the fp64 oracle: the columns must match
exactly (same ranking: value descending, then the smaller column), the shares within the row
softmax tolerance."""
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


def check(x, k, what):
    v, i, l = binding.osm_softmax_topk(x.cuda(), k)
    torch.cuda.synchronize()
    vr, ir, lr = oracle.softmax_topk(x.numpy(), k)
    i = i.cpu().numpy().astype(np.int64)
    assert np.array_equal(i, ir), f"{what}: columns differ in {np.sum(i != ir)} places"
    v = v.cpu().numpy().astype(np.float64)
    dv = np.abs(v - vr).max()
    assert dv <= parity.SOFTMAX_Y_ATOL, f"{what}: max|dvalue| = {dv:.3e}"
    l = l.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lr)
    assert np.array_equal(np.isfinite(l), fin), what
    if fin.any():
        dl = (np.abs(l[fin] - lr[fin]) / np.maximum(1.0, np.abs(lr[fin]))).max()
        assert dl <= parity.SOFTMAX_LSE_RTOL, f"{what}: max rel|dlse| = {dl:.3e}"


# (rows, cols, k): warp-per-row and CTA-per-row paths, 16-byte and scalar loads, every list size
CASES = [(64, 4000, 8), (33, 4001, 5), (7, 100000, 32), (100, 50, 1), (10, 4096, 16),
         (9, 4097, 32), (5, 9000, 2), (300, 128, 4), (3, 33, 32), (2, 1, 1), (11, 262144, 12),
         # rows staged in shared memory: many rows per warp (the ring wraps), the widest row,
         # rows shorter than a warp's loads
         (40000, 128, 3), (5000, 1024, 9), (37, 4096, 32), (129, 12, 2),
         # long rows staged in segments shared by the warps of a CTA: a partial last segment,
         # several rows per CTA
         (40, 12300, 7), (2000, 4100, 16)]


@pytest.mark.parametrize("rows,cols,k", CASES, ids=lambda x: str(x))
def test_topk_parity(rows, cols, k):
    x = inputs.softmax_inputs(rows, cols, seed=9000 + rows + cols + k)
    check(x, k, f"{(rows, cols, k)}")


@pytest.mark.parametrize("cols", [300, 5000])
def test_topk_ties_and_masked_rows(cols):
    """Integer-valued rows (many ties: the smaller column must win), rows of -inf with a few
    finite entries, a fully -inf row and the overflow row."""
    g = torch.Generator().manual_seed(31 + cols)
    x = torch.randint(-4, 5, (12, cols), generator=g).to(torch.float32)
    x[2] = -float("inf")
    x[2, cols // 2] = 7.0
    x[3] = -float("inf")                     # nothing finite: shares 0, lse -inf
    x[4, :] = 1000.0
    x[4, :3] = torch.tensor([1000.0, 1001.0, 1002.0])
    x[5] = 3.0                               # a constant row: columns 0..k-1
    for k in (1, 7, 32):
        check(x, k, f"ties cols={cols} k={k}")


def test_topk_full_size_workloads():
    """The bench's workloads at full size: every row's columns and shares on seeded samples of
    rows (the oracle sorts each sampled row)."""
    for w in inputs.TOPK_WORKLOADS.values():
        x = inputs.softmax_inputs(w.rows, w.cols, w.seed, w.std, w.spike)
        v, i, l = binding.osm_softmax_topk(x.cuda(), w.k)
        torch.cuda.synchronize()
        g = torch.Generator().manual_seed(w.seed + 5)
        rows = torch.randperm(w.rows, generator=g)[:256].sort().values.numpy()
        vr, ir, lr = oracle.softmax_topk(x[rows].numpy(), w.k)
        assert np.array_equal(i.cpu().numpy()[rows].astype(np.int64), ir), w.name
        assert np.abs(v.cpu().numpy()[rows] - vr).max() <= parity.SOFTMAX_Y_ATOL, w.name
        lg = l.cpu().numpy()[rows].astype(np.float64)
        assert (np.abs(lg - lr) / np.maximum(1.0, np.abs(lr))).max() <= parity.SOFTMAX_LSE_RTOL


# k > 32: a CTA per row, a floor and a candidate buffer (short and long rows, k up to the largest
# supported; each thread keeps its 1, 2 or 4 largest values as k crosses 256 and 512; 16-byte
# and 4-byte loads; several chunks per row)
LARGE_K = [(64, 4000, 33), (16, 32000, 100), (5, 131072, 64), (40, 300, 257), (3, 5000, 1024),
           (200, 64, 64), (2, 1024, 1024), (3, 131072, 1024), (4, 65536, 512), (4, 65536, 513),
           (4, 100003, 300), (6, 70001, 40),
           # many rows per CTA, a row of 8196 columns, k = 129 and 256 (two values per thread)
           (2000, 8196, 40), (7, 16384, 256), (3, 12288, 129), (600, 8192, 33)]


@pytest.mark.parametrize("rows,cols,k", LARGE_K, ids=lambda x: str(x))
def test_topk_large_k_parity(rows, cols, k):
    x = inputs.softmax_inputs(rows, cols, seed=9300 + rows + cols + k)
    check(x, k, f"{(rows, cols, k)}")


@pytest.mark.parametrize("cols", [300, 5000, 20000])
def test_topk_large_k_ties_and_masked_rows(cols):
    """The tie rule (the smaller column first) at the k-th place decides which of many equal
    values are kept; rows of -inf, a constant row, the overflow row.  At 20000 columns the rows
    with more entries at the floor than the candidate buffer holds (constant, nearly constant,
    fewer than k finite values) take the exact radix route."""
    g = torch.Generator().manual_seed(71 + cols)
    x = torch.randint(-4, 5, (12, cols), generator=g).to(torch.float32)
    x[2] = -float("inf")
    x[2, cols // 2] = 7.0
    x[3] = -float("inf")
    x[4, :] = 1000.0
    x[4, :3] = torch.tensor([1000.0, 1001.0, 1002.0])
    x[5] = 3.0
    x[6, ::2] = -0.0                          # -0 and +0 are equal values
    x[6, 1::2] = 0.0
    for k in (33, 100, 299):
        check(x, k, f"ties cols={cols} k={k}")


@pytest.mark.parametrize("cols", [65536, 65537])
def test_topk_large_k_sorted_and_trending_rows(cols):
    """Rows in ascending order beat every running floor, so the candidate buffer overflows
    during the one-read sweep and the row is read once more against the final floor; rows in
    descending order meet their floor at once; rows that rise slowly under noise push the
    buffer past half full, so that entries below the floors are dropped during the sweep."""
    x = inputs.softmax_inputs(12, cols, seed=9401 + cols)
    x[:4] = x[:4].sort(dim=1).values
    x[4:8] = x[4:8].sort(dim=1, descending=True).values
    x[8:] += torch.linspace(0.0, 60.0, cols)
    for k in (40, 100, 600):
        check(x, k, f"sorted cols={cols} k={k}")
