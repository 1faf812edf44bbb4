"""Pins of the oracle's Philox4x32-10 and uniform construction (CPU).

The pages name no generator; the verify step draws its uniforms from Philox4x32-10 (Salmon et al.,
SC'11). The oracle's implementation is pinned against a *call* to curand's host-side
Philox4x32-10 generator, whose j-th output block is Philox4x32-10(counter = (0, 0, j, 0), key = seed).
That exercises the full key, counter word 2 and every round; the other counter words are pinned on the
GPU against curand's device ``curand_Philox4x32_10(counter, key)``.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle

CURAND = "/usr/local/cuda/lib64/libcurand.so"


def _curand_host_blocks(seed: int, nblocks: int) -> np.ndarray:
    cr = ctypes.CDLL(CURAND)
    gen = ctypes.c_void_p()
    assert cr.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(4 * nblocks, dtype=np.uint32)
        assert cr.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                 ctypes.c_size_t(out.size)) == 0
    finally:
        cr.curandDestroyGenerator(gen)
    return out.reshape(nblocks, 4)


@pytest.mark.skipif(not os.path.exists(CURAND), reason="libcurand not installed")
@pytest.mark.parametrize("seed", [0, 1, 1234, 0x0123456789ABCDEF, 2**64 - 1])
def test_philox_matches_curand_host_generator(seed):
    blocks = _curand_host_blocks(seed, 2048)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for j in range(0, 2048, 1 if seed in (0, 1234) else 7):
        got = oracle.philox4x32_10([0, 0, j, 0], key)
        assert np.array_equal(got, blocks[j]), (seed, j)


def test_uniform_is_top_24_bits_of_word0():
    for seed, step, b, slot, purpose in [(0, 0, 0, 0, 0), (1234, 7, 3, 5, 1), (2**63 + 5, 2**40 + 3, 99, 31, 0)]:
        ctr = [step & 0xFFFFFFFF, step >> 32, b, (slot << 8) | purpose]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        x0 = int(oracle.philox4x32_10(ctr, key)[0])
        u = oracle.uniform(seed, step, b, slot, purpose)
        assert u == (x0 >> 8) / 2.0**24
        assert 0.0 <= u <= 1.0 - 2.0**-24
        assert float(np.float32(u)) == u  # exactly representable in fp32 as well


def test_uniform_changes_with_every_key_field():
    base = oracle.uniform(1234, 5, 6, 2, 0)
    others = [oracle.uniform(1235, 5, 6, 2, 0), oracle.uniform(1234 + (1 << 32), 5, 6, 2, 0),
              oracle.uniform(1234, 6, 6, 2, 0), oracle.uniform(1234, 5 + (1 << 32), 6, 2, 0),
              oracle.uniform(1234, 5, 7, 2, 0), oracle.uniform(1234, 5, 6, 3, 0),
              oracle.uniform(1234, 5, 6, 2, 1)]
    assert all(o != base for o in others)


def test_uniform_distribution_is_flat():
    us = np.array([oracle.uniform(99, s, b, 0, 0) for s in range(50) for b in range(400)])
    hist, _ = np.histogram(us, bins=20, range=(0, 1))
    from scipy.stats import chisquare
    assert chisquare(hist).pvalue > 1e-4
