"""The fp64 oracle against its pins (no GPU)."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default_oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    x = np.zeros((1, 4, 1, 2))
    with pytest.raises(ValueError):   # cu_seqlens not ending at T
        orc.recurrent(x, x, x, x, np.zeros((1, 4, 1)), 1.0, cu_seqlens=np.array([0, 3], np.int32))
    with pytest.raises(ValueError):   # decreasing offsets
        orc.chunkwise(x, x, x, x, np.zeros((1, 4, 1)), 1.0, 2,
                      cu_seqlens=np.array([0, 3, 2, 4], np.int32))
