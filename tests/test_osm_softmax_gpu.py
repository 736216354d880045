"""osm_softmax on the GPU, through the C ABI, against the fp64 oracle."""
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


def run_gpu(x, misalign=False):
    rows, cols = x.shape
    if misalign:  # start the rows 4 bytes past a 16-byte boundary: scalar path
        buf = torch.empty(rows * cols + 1, dtype=torch.float32, device="cuda")
        xd = buf[1:].view(rows, cols)
        xd.copy_(x)
        out = torch.empty(rows * cols + 1, dtype=torch.float32, device="cuda")[1:].view(rows, cols)
    else:
        xd = x.cuda()
        out = None
    y, lse = binding.osm_softmax(xd, out=out)
    torch.cuda.synchronize()
    return y.cpu().numpy(), lse.cpu().numpy()


SHAPES = [(1, 1), (3, 5), (7, 128), (7, 129), (64, 1000), (5, 1024), (5, 1025), (3, 2048),
          (3, 4000), (3, 4096), (3, 8191), (2, 16384), (2, 16385), (2, 40000), (300, 64)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("misalign", [False, True])
def test_softmax_parity(rows, cols, misalign):
    x = inputs.softmax_inputs(rows, cols, seed=rows * 7 + cols, std=9.0, spike=100.0)
    y, lse = run_gpu(x, misalign)
    yref, lref = oracle.softmax_rows(x.numpy())
    parity.check_softmax(y, lse, yref, lref, f"{rows}x{cols} misalign={misalign}")


def test_softmax_full_size_sampled():
    w = inputs.SOFTMAX_WORKLOADS["softmax_65536x4000"]
    x = inputs.softmax_workload_inputs(w)
    xd = x.cuda()
    y, lse = binding.osm_softmax(xd)
    torch.cuda.synchronize()
    sums = y.double().sum(dim=1)
    assert torch.isfinite(y).all() and (y >= 0).all()
    assert (sums - 1.0).abs().max().item() <= parity.SOFTMAX_SUM_ATOL
    g = torch.Generator().manual_seed(5)
    rows = torch.randperm(w.rows, generator=g)[:2048].sort().values
    rows[0] = 0
    rows[-1] = w.rows - 1
    yref, lref = oracle.softmax_rows(x[rows].numpy())
    parity.check_softmax(y[rows.cuda()].cpu().numpy(), lse[rows.cuda()].cpu().numpy(), yref, lref,
                         "softmax_65536x4000")


def test_softmax_special_rows():
    x = torch.tensor([
        [1000.0, 1001.0, 1002.0, -np.inf],
        [-np.inf, -np.inf, -np.inf, -np.inf],
        [-np.inf, -np.inf, 1.0, 2.0],
        [88.7, 88.8, -88.8, 0.0],
    ], dtype=torch.float32)
    y, lse = run_gpu(x)
    yref, lref = oracle.softmax_rows(x.numpy())
    assert np.all(y[1] == 0.0) and lse[1] == -np.inf
    parity.check_softmax(y, lse, yref, lref, "special rows")
    t = np.exp(np.array([-2.0, -1.0, 0.0]))
    assert np.abs(y[0, :3] - t / t.sum()).max() < 1e-6


def test_softmax_in_place_and_no_lse():
    x = inputs.softmax_inputs(33, 4000, seed=3)
    yref, _ = oracle.softmax_rows(x.numpy())
    xd = x.cuda()
    y, lse = binding.osm_softmax(xd, out=xd, return_lse=False)
    torch.cuda.synchronize()
    assert lse is None and y.data_ptr() == xd.data_ptr()
    assert np.abs(y.cpu().numpy() - yref).max() <= parity.SOFTMAX_Y_ATOL
