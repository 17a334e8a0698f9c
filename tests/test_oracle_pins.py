"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

from oracle import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_thread_count_does_not_change_bits(oracle_lib):
    rng = np.random.default_rng(3)
    lens = [9, 31, 4]
    T, H, dk, dv = sum(lens), 3, 8, 8
    q, k, v = (rng.standard_normal((T, H, n)) for n in (dk, dk, dv))
    g = -np.abs(rng.standard_normal((T, H, dk)))
    beta = rng.uniform(0, 1, (T, H))
    cu = np.concatenate([[0], np.cumsum(lens)])
    a = oracle.run(q, k, v, g, beta, cu, threads=1, lib=oracle_lib)
    b = oracle.run(q, k, v, g, beta, cu, threads=5, lib=oracle_lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_snapshot_at_zero_and_end(oracle_lib):
    rng = np.random.default_rng(4)
    T, dk, dv = 6, 3, 3
    q, k, v = (rng.standard_normal((T, 1, n)) for n in (dk, dk, dv))
    g = -np.abs(rng.standard_normal((T, 1, dk)))
    beta = rng.uniform(0, 1, (T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, S, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=[0, T, T + 5], lib=oracle_lib)
    assert np.array_equal(snaps[0], S0)
    assert np.array_equal(snaps[1], S)
    assert np.isnan(snaps[2]).all()


def test_rejects_non_monotone_cu_seqlens(oracle_lib):
    z = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.run(z, z, z, z, np.zeros((4, 1)), [0, 3, 2, 4], lib=oracle_lib)


def test_empty_sequences(oracle_lib):
    rng = np.random.default_rng(5)
    S0 = rng.standard_normal((2, 1, 2, 2))
    z = np.zeros((0, 1, 2))
    o, S, _ = oracle.run(z, z, z, z, np.zeros((0, 1)), [0, 0, 0], S0=S0, lib=oracle_lib)
    assert o.shape == (0, 1, 2)
    assert np.array_equal(S, S0)
