"""Tolerances and comparison helpers shared by the GPU parity tests.

Attention: max |O_gpu - O_oracle| <= 1e-2 (bf16 output, fp32 accumulation) and
|LSE_gpu - LSE_oracle| <= 1e-3 * max(1, |LSE_oracle|) (relative, with an absolute floor of
1e-3 where LSE is near 0).
Row softmax: max |y_gpu - y_oracle| <= 1e-6, |sum_j y_ij - 1| <= 1e-5 per row,
|lse_gpu - lse_oracle| <= 1e-5 * max(1, |lse_oracle|).
"""
import numpy as np

ATTN_O_ATOL = 1e-2
ATTN_LSE_RTOL = 1e-3
SOFTMAX_Y_ATOL = 1e-6
SOFTMAX_SUM_ATOL = 1e-5
SOFTMAX_LSE_RTOL = 1e-5


def check_attention(O, L, Oref, Lref, what=""):
    O = np.asarray(O, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    assert O.shape == Oref.shape and L.shape == Lref.shape, what
    assert np.isfinite(O).all(), f"{what}: non-finite O"
    assert np.isfinite(L).all(), f"{what}: non-finite LSE"
    dO = np.abs(O - Oref).max() if O.size else 0.0
    dL = (np.abs(L - Lref) / np.maximum(1.0, np.abs(Lref))).max() if L.size else 0.0
    assert dO <= ATTN_O_ATOL, f"{what}: max|dO| = {dO:.3e}"
    assert dL <= ATTN_LSE_RTOL, f"{what}: max rel|dLSE| = {dL:.3e}"
    return dO, dL


def check_softmax(y, lse, yref, lseref, what=""):
    y = np.asarray(y, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    dy = np.abs(y - yref).max() if y.size else 0.0
    assert dy <= SOFTMAX_Y_ATOL, f"{what}: max|dy| = {dy:.3e}"
    fin = np.isfinite(lseref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    if fin.any():
        dl = (np.abs(lse[fin] - lseref[fin]) / np.maximum(1.0, np.abs(lseref[fin]))).max()
        assert dl <= SOFTMAX_LSE_RTOL, f"{what}: max rel|dlse| = {dl:.3e}"
    assert np.array_equal(lse[~fin], lseref[~fin]), f"{what}: -inf lse rows differ"
    sums = y.sum(axis=1)
    rows_ok = fin
    if rows_ok.any():
        ds = np.abs(sums[rows_ok] - 1.0).max()
        assert ds <= SOFTMAX_SUM_ATOL, f"{what}: max|sum-1| = {ds:.3e}"
    return dy


def check_attention_allow_empty(O, L, Oref, Lref, what=""):
    """As check_attention, but rows with no allowed key (Lref = -inf) must be exactly O = 0 and
    LSE = -inf."""
    O = np.asarray(O, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    empty = np.isneginf(Lref)
    assert np.array_equal(np.isneginf(L), empty), f"{what}: empty rows differ"
    assert np.all(O[empty] == 0.0), f"{what}: empty rows are not zero"
    if (~empty).any():
        check_attention(O[~empty], L[~empty], Oref[~empty], Lref[~empty], what)
