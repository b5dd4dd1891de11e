"""The fp64 oracle against what the sources and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(None)


def test_threads_match_single_thread():
    """Threading over (sequence, head) pairs changes nothing."""
    rng = np.random.default_rng(5)
    B, T, H, d = 3, 4, 2, 128
    n = rng.standard_normal
    args = dict(q=n((B, T, H, d)), k=n((B, T, H, d)), v=n((B, T, H, d)), z=n((B, T, H, d)),
                beta_logit=n((B, T, H)), gate_logit=n((B, T, H, d)),
                conv_w=0.25 * n((3, H * d, 4)), dt_bias=0.1 * n((H, d)),
                A_log=rng.uniform(-4, 0, (H, d)), gamma=1 + 0.1 * n((H, d)),
                conv_state=n((B, 3, 3 * H * d)), S=0.01 * n((B, H, d, d)))
    a = oracle.run(**args, nthreads=1)
    b = oracle.run(**args, nthreads=4)
    for x, y in ((a.o, b.o), (a.S, b.S), (a.conv_state, b.conv_state)):
        assert np.array_equal(x, y)


def test_empty_inputs():
    d, H = 128, 1
    z4 = np.zeros((1, 0, H, d))
    out = oracle.run(z4, z4, z4, z4, np.zeros((1, 0, H)), z4, np.zeros((3, H * d, 4)),
                     np.zeros((H, d)), np.zeros((H, d)), np.ones((H, d)),
                     np.ones((1, 3, 3 * H * d)), np.ones((1, H, d, d)))
    assert out.o.shape == (1, 0, H, d)
    assert np.all(out.S == 1) and np.all(out.conv_state == 1)


def test_cpu_count():
    assert oracle.cpu_count() >= 1
