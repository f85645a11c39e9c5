"""Pins for the oracle's Philox4x32-10 stream and its uniform mapping.

The generator is pinned against an independent implementation: cuRAND's host
PHILOX4_32_10 generator (a library routine run on the CPU).  With seed s the
host generator uses key (s mod 2^32, s >> 32) and emits the four words of
block i = 0, 1, 2, ... from counter (0, 0, i, 0).
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def _load_curand():
    cands = [ctypes.util.find_library("curand"), "libcurand.so", "libcurand.so.10",
             "/usr/local/cuda/lib64/libcurand.so"]
    for c in cands:
        if not c:
            continue
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


def _curand_words(lib, seed, n):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return out
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 2 ** 64 - 1, 0xDEADBEEF00000000])
def test_philox_matches_curand_host_generator(seed):
    lib = _load_curand()
    if lib is None:
        pytest.skip("libcurand not available")
    n = 8192
    ref = _curand_words(lib, seed, n)
    ctr = np.zeros((n // 4, 4), dtype=np.int64)
    ctr[:, 2] = np.arange(n // 4)
    ours = philox.philox4x32_10(ctr, philox.seed_key(seed)).reshape(-1)
    assert np.array_equal(ours, ref)


def test_philox_key_and_counter_words_all_matter():
    base = philox.philox4x32_10(np.array([[5, 6, 7, 8]]), (9, 10))
    for w in range(4):
        c = np.array([[5, 6, 7, 8]])
        c[0, w] ^= 1
        assert not np.array_equal(philox.philox4x32_10(c, (9, 10)), base)
    assert not np.array_equal(philox.philox4x32_10(np.array([[5, 6, 7, 8]]), (9, 11)), base)


def test_uniform_mapping_exact_in_float32_and_open_interval():
    rng = np.random.default_rng(0)
    w = np.concatenate([np.array([0, 1, 511, 512, 2 ** 32 - 1], dtype=np.uint64),
                        rng.integers(0, 2 ** 32, 100000, dtype=np.uint64)])
    u = philox.uniform_from_word(w)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    om = philox.one_minus_uniform_from_word(w)
    assert np.array_equal(om + u, np.ones_like(u))
    assert u.min() == 0.5 * 2.0 ** -23
    assert u.max() == 1 - 0.5 * 2.0 ** -23


def test_accept_stream_is_uniform():
    us = np.array([philox.accept_uniform(7, r, j) for r in range(2000) for j in range(4)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    assert abs(us.mean() - 0.5) < 5 * np.sqrt(1 / 12 / len(us))


def test_race_exponentials_are_exp1_and_uncorrelated():
    v = np.arange(200000)
    E = philox.race_exponentials(123, 3, 1, v)
    assert stats.kstest(E, "expon").pvalue > 1e-3
    assert abs(np.corrcoef(E[:-1], E[1:])[0, 1]) < 0.01
    # a different position or row gives a different stream
    assert not np.array_equal(E[:64], philox.race_exponentials(123, 3, 2, v[:64]))
    assert not np.array_equal(E[:64], philox.race_exponentials(123, 4, 1, v[:64]))


def test_race_exponential_precise_near_one():
    # The largest uniform 1 - 2^-24 must give E = 2^-24 to full relative precision.
    w = np.array([2 ** 32 - 1], dtype=np.uint64)
    om = philox.one_minus_uniform_from_word(w)
    E = -np.log1p(-om)
    assert abs(E[0] / 2.0 ** -24 - 1) < 1e-7
