"""Pins of the oracle's random numbers (CPU only).

Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
SC'11) is checked against an independent implementation: cuRAND's host-side
PHILOX4_32_10 generator, a library routine that runs on the CPU.  Its output
stream, for seed S and output offset o, is block g = o / 4 of
Philox(counter = (g >> 16, g >> 48, g & 0xffff, 0), key = (S low, S high)),
so counter words 0, 1 and 2, the key schedule, both round multipliers and the
output word order are all exercised.  Counter word 3 is checked against
cuRAND's device generator in the GPU tests.
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

import oracle

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def _curand():
    cands = []
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        cands.append(os.path.join(cuda_home, sub, "libcurand.so"))
    found = ctypes.util.find_library("curand")
    if found:
        cands.append(found)
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not available")


def _host_stream(lib, seed, n, offset=0):
    gen = ctypes.c_void_p()
    st = lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10)
    if st != 0:
        pytest.skip(f"curandCreateGeneratorHost failed ({st})")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


def _key(seed):
    return [seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF]


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF, 2**32 + 7])
def test_philox_matches_curand_host_stream(seed):
    lib = _curand()
    n_blocks = 300
    h = _host_stream(lib, seed, 4 * n_blocks).reshape(n_blocks, 4)
    for g in range(n_blocks):
        got = oracle.philox4x32_10([0, 0, g, 0], _key(seed))
        assert list(got) == list(h[g]), (seed, g)


@pytest.mark.parametrize("block", [1 << 16, (1 << 16) * 3 + 5, 1 << 48, (1 << 48) * 5 + (7 << 16) + 9,
                                   (0x3FFF << 48) + (0xABCDE << 16) + 0x1234])
def test_philox_counter_words_0_and_1(block):
    lib = _curand()
    seed = 0x9E3779B97F4A7C15
    h = _host_stream(lib, seed, 4, offset=4 * block)
    ctr = [(block >> 16) & 0xFFFFFFFF, (block >> 48) & 0xFFFFFFFF, block & 0xFFFF, 0]
    assert list(oracle.philox4x32_10(ctr, _key(seed))) == list(h)


def test_uniform_map_closed_form():
    # U(w) = ((w >> 9) + 1/2) 2^-23: endpoints, exactness and monotonicity.
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(511) == 2.0 ** -24  # the low 9 bits are dropped
    assert oracle.uniform(512) == 3 * 2.0 ** -24
    rng = np.random.default_rng(0)
    ws = np.sort(rng.integers(0, 2**32, size=2000, dtype=np.uint64))
    us = [oracle.uniform(int(w)) for w in ws]
    assert all(0.0 < u < 1.0 for u in us)
    assert all(a <= b for a, b in zip(us, us[1:]))
    for w, u in zip(ws[:200], us[:200]):
        k = u * 2.0 ** 24
        assert k == int(k) and int(k) % 2 == 1  # an odd multiple of 2^-24
        assert np.float32(u) == u  # exact in fp32 too


def test_draws_are_uniform_ks():
    # The acceptance draws over many requests are U(0, 1) (Kolmogorov-Smirnov).
    from scipy import stats

    us = [oracle.uniform(oracle.draw(0, b, 0, 0, 0)) for b in range(20000)]
    assert stats.kstest(us, "uniform").pvalue > 1e-4
