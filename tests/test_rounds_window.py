"""The library's cosine-window host function (spec_anyorder_window) against
the oracle's (Self-Speculative Masked Diffusions, key design 4), on a grid;
both run on the host, so no GPU is needed.  dtau values are exact in fp32
(the C ABI takes a float)."""
import numpy as np
import pytest

import oracle
import rejection_sampling_gb300 as rs


@pytest.fixture(scope="module", autouse=True)
def _libs():
    oracle.build()
    rs.build()
    rs.load()


@pytest.mark.parametrize("D", [1, 2, 37, 256, 1000])
@pytest.mark.parametrize("dtau", [0.0, 0.0078125, 0.05, 0.083, 0.25, 1.0, 2.0])
def test_window_matches_the_oracle(D, dtau):
    dt = float(np.float32(dtau))
    for i in list(range(min(D, 300))) + [D - 1, D, D + 5]:
        if i < 0:
            continue
        assert rs.spec_anyorder_window(D, i, dt) == oracle.cosine_window(D, i, dt), (D, i, dt)


def test_window_bad_arguments():
    assert rs.spec_anyorder_window(0, 0, 0.1) == -1
    assert rs.spec_anyorder_window(10, -1, 0.1) == -1
    assert rs.spec_anyorder_window(10, 10, 0.1) == 0
