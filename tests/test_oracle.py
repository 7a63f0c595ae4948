"""The fp64 oracle against facts independent of it (CPU only)."""

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_oracle_rejects_bad_inputs(oracle_lib):
    lens = [20, 3]
    qbits, Kc, Vc = P.dense_case(2, 4, 2, lens, seed=5)
    kc, vc, tb, ln = P.scatter_pages(Kc, Vc, lens, 16, seed=5)
    bad = tb.copy()
    bad[0, 1] = kc.shape[0]          # block id == num_blocks
    with pytest.raises(oracle.OracleError, match="block id"):
        P.run(oracle_lib, qbits, kc, vc, bad, ln, 0.1, 0.05, 0.05)
    too_long = ln.copy()
    too_long[1] = tb.shape[1] * 16 + 1
    with pytest.raises(oracle.OracleError, match="seq_len"):
        P.run(oracle_lib, qbits, kc, vc, tb, too_long, 0.1, 0.05, 0.05)
    with pytest.raises(oracle.OracleError, match="seq id"):
        P.run(oracle_lib, qbits, kc, vc, tb, ln, 0.1, 0.05, 0.05, seq_ids=[2])


def test_oracle_seq_subset_matches_full(oracle_lib):
    lens = [20, 3, 47, 16]
    qbits, Kc, Vc = P.dense_case(4, 8, 2, lens, seed=6)
    kc, vc, tb, ln = P.scatter_pages(Kc, Vc, lens, 16, seed=6)
    full = P.run(oracle_lib, qbits, kc, vc, tb, ln, 0.1, 0.05, 0.05)
    sub = P.run(oracle_lib, qbits, kc, vc, tb, ln, 0.1, 0.05, 0.05, seq_ids=[3, 0])
    assert np.array_equal(sub, full[[3, 0]])


def test_oracle_thread_count_does_not_change_result(oracle_lib):
    lens = [100, 37, 64]
    qbits, Kc, Vc = P.dense_case(3, 8, 1, lens, seed=7)
    kc, vc, tb, ln = P.scatter_pages(Kc, Vc, lens, 16, seed=7)
    a = P.run(oracle_lib, qbits, kc, vc, tb, ln, 0.1, 0.05, 0.05, num_threads=1)
    b = P.run(oracle_lib, qbits, kc, vc, tb, ln, 0.1, 0.05, 0.05, num_threads=4)
    assert np.array_equal(a, b)
