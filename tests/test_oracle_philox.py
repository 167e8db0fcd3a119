"""Pins for the oracle's counter-based uniforms.

The oracle's Philox4x32-10 block function (Salmon et al., SC'11) is checked
against an independent implementation: cuRAND's *host* generator
(CURAND_RNG_PSEUDO_PHILOX4_32_10, run on the CPU, no GPU needed). With seed S
that generator emits, at output offset o, word (o mod 4) of
Philox(key = (S_lo, S_hi), counter = (c_lo, c_hi, s, 0)) where
s = (o div 4) mod 65536 and c = (o div 4) div 65536 -- which covers every
counter word the verify step uses: (sequence b, position i, purpose, 0).
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def _curand():
    cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcurand.so"),
             ctypes.util.find_library("curand")]
    for c in cands:
        if c and (os.path.exists(c) or not os.path.isabs(c)):
            try:
                return ctypes.CDLL(c)
            except OSError:
                pass
    pytest.skip("libcurand not available")


def _curand_words(lib, seed, offset, n=4):
    g = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(g), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(g, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, np.uint32)
        assert lib.curandGenerate(g, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return [int(v) for v in out]
    finally:
        lib.curandDestroyGenerator(g)


def _offset(c0, c1, c2):
    return 4 * ((c0 + (c1 << 32)) * 65536 + c2)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 2**64 - 1, 987654321])
def test_philox_matches_curand_host_generator(oracle_mod, seed):
    lib = _curand()
    key = (seed & 0xFFFFFFFF, seed >> 32)
    rng = np.random.default_rng(seed % 1000)
    counters = [(0, 0, 0), (0, 1, 0), (0, 1, 1), (511, 7, 1), (255, 10, 0), (3, 0, 1),
                (2**32 - 1, 5, 0), (12345, 4095, 1)]  # offsets must fit 64 bits
    counters += [(int(rng.integers(0, 1 << 20)), int(rng.integers(0, 64)), int(rng.integers(0, 2)))
                 for _ in range(8)]
    for (b, i, purpose) in counters:
        want = _curand_words(lib, seed, _offset(b, i, purpose))
        got = list(oracle_mod.philox4x32_10((b, i, purpose, 0), key))
        assert got == want, (seed, b, i, purpose)


def test_seeded_uniforms_use_the_documented_counter(oracle_mod):
    lib = _curand()
    seed = 0xDEADBEEF12345678
    for b, i in [(0, 1), (7, 3), (300, 11)]:
        w_acc = _curand_words(lib, seed, _offset(b, i, 0))
        w_drw = _curand_words(lib, seed, _offset(b, i, 1))
        assert oracle_mod.accept_uniform(seed, b, i) == (2 * (w_acc[0] >> 9) + 1) * 2.0**-24
        k = (w_drw[0] << 20) | (w_drw[1] >> 12)
        assert oracle_mod.draw_uniform(seed, b, i) == (2 * k + 1) * 2.0**-53


def test_u24_u52_are_exact_dyadics_inside_the_unit_interval(oracle_mod):
    assert oracle_mod.u24(0) == 2.0**-24
    assert oracle_mod.u24(0xFFFFFFFF) == 1.0 - 2.0**-24
    assert oracle_mod.u52(0, 0) == 2.0**-53
    assert oracle_mod.u52(0xFFFFFFFF, 0xFFFFFFFF) == 1.0 - 2.0**-53
    rng = np.random.default_rng(5)
    for x in rng.integers(0, 2**32, 200):
        u = oracle_mod.u24(int(x))
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u          # exact in fp32 as well
        assert (u * 2**24) % 2 == 1               # odd multiple of 2^-24
    xs = np.sort(rng.integers(0, 2**32, 100))
    us = [oracle_mod.u24(int(x)) for x in xs]
    assert all(a <= b for a, b in zip(us, us[1:]))


def test_seeded_uniforms_are_uniform(oracle_mod):
    # Kolmogorov-Smirnov distance over many counters; a broken mapping
    # (e.g. a wrong shift) shows up as a large deviation.
    from scipy import stats
    us = np.array([oracle_mod.accept_uniform(42, b, 1 + (b % 9)) for b in range(20000)])
    assert stats.kstest(us, "uniform").pvalue > 1e-4
    ds = np.array([oracle_mod.draw_uniform(42, b, 1 + (b % 9)) for b in range(20000)])
    assert stats.kstest(ds, "uniform").pvalue > 1e-4
