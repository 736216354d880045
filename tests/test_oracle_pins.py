"""The fp64 oracle against the pages' worked examples, closed forms, a library routine,
40-digit brute force and the method's invariants (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np

    q = np.zeros((1, 1, 4, 2), dtype=np.uint16)
    with pytest.raises(ValueError):
        orc.attention(q, q, q, 1.0, False, rows=np.array([4]))
    with pytest.raises(ValueError):
        orc.attention(q, q, q, 1.0, False, rows=np.array([-1]))
    with pytest.raises(TypeError):
        orc.attention(q.astype(np.float32), q, q, 1.0, False)


def test_oracle_row_subset_matches_full(orc):
    from online_softmax_tiled_attn_gb300 import inputs
    import numpy as np

    q, k, v = inputs.attn_inputs(2, 2, 33, 8, seed=21)
    O, L = orc.attention(q, k, v, 0.35, True)
    rows = np.array([0, 5, 32, 33, 70, 131])
    Os, Ls = orc.attention(q, k, v, 0.35, True, rows=rows)
    assert np.array_equal(Os, O.reshape(-1, 8)[rows])
    assert np.array_equal(Ls, L.reshape(-1)[rows])
