"""The fp64 oracle against its pins (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
from tests.pins import PINS, _rand_chunk

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, lib):
    pin(lib)


def test_fp16_stored_T_error_order(lib):
    """§4 error table: storing T in fp16 costs a relative error of order 5.72e-5."""
    with open(os.path.join(GOLDEN, "paper_counts.json")) as f:
        ref = json.load(f)["inverse_errors"]["fp16_T_relative"]
    rng = np.random.default_rng(21)
    rel = []
    for _ in range(50):
        k, v, beta = _rand_chunk(rng, 32, 128, 1)
        T, _, _, _ = oracle.oracle_chunk(k, v, beta, 32, lib=lib)
        T16 = T.astype(np.float16).astype(np.float64)
        rel.append(np.abs(T16 - T).max() / np.abs(T).max())
    assert ref / 3 <= np.mean(rel) <= ref * 3, np.mean(rel)


def test_bad_arguments(lib):
    with pytest.raises(ValueError):
        oracle.oracle_chunk(np.zeros((5, 4)), np.zeros((5, 4)), np.zeros(5), 4, lib=lib)
    k = np.zeros((1, 10, 1, 4))
    with pytest.raises(ValueError):  # cu_seqlens must end at the token count
        oracle.oracle_fwd(k, k, np.zeros((1, 10, 1)), 4, cu_seqlens=[0, 3, 9], lib=lib)
    with pytest.raises(ValueError):  # and be nondecreasing
        oracle.oracle_fwd(k, k, np.zeros((1, 10, 1)), 4, cu_seqlens=[0, 6, 3, 10], lib=lib)


def test_empty_sequences(lib):
    """Zero-length sequences in a packed batch produce no rows and disturb nothing."""
    rng = np.random.default_rng(22)
    k = rng.standard_normal((1, 9, 1, 4))
    beta = rng.uniform(0.1, 0.9, (1, 9, 1))
    To, Wo, Uo = oracle.oracle_fwd(k, k, beta, 4, cu_seqlens=[0, 0, 5, 5, 9], lib=lib)
    Ta, Wa, Ua = oracle.oracle_fwd(k, k, beta, 4, cu_seqlens=[0, 5, 9], lib=lib)
    np.testing.assert_array_equal(To, Ta)
    np.testing.assert_array_equal(Wo, Wa)
