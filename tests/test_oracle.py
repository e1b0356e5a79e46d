"""The CPU oracle against its pins (no GPU)."""

import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(oracle.lib())


def test_oracle_rejects_bad_input():
    import numpy as np
    from oracle_pins import contiguous, index_case, mla_case
    c = index_case(n=8, pos=8)           # position == context length
    with pytest.raises(ValueError, match="position"):
        oracle.index_scores(c["q"], c["w"], c["ssmax_s"], c["ssmax_b"], None, c["q_seq"], c["q_pos"], c["keys"],
                            contiguous([8], 8))
    q, lat, lay = mla_case(n=5)
    with pytest.raises(ValueError, match="index"):
        oracle.sparse_mla(q, lat, lay, 0, np.array([5], np.int32), 1, 1.0)
    bad = oracle.Layout(np.array([5], np.int32), 5, page_table=np.array([[3]], np.int32), page_size=4)
    with pytest.raises(ValueError, match="page"):
        oracle.sparse_mla(q, lat, bad, 0, np.array([1], np.int32), 1, 1.0)
