"""Pins of the oracle's Philox4x32-10 and of stochastic rounding.

Philox (Salmon et al., SC'11) is pinned against cuRAND's host-side
PHILOX4_32_10 generator, which runs on the CPU.  With seed s, its output
block b (words 4b .. 4b+3) is Philox4x32-10(counter = (q lo, q hi, b mod 2^16, 0),
key = (s lo, s hi)) with q = b div 2^16, so the pin covers both key words and
counter words 0, 1 and 2.  SR (Format-Aware Fusion for Fast FP4 Pretraining,
Sec. 2.5, Eq. 9) is pinned by its defining statistics.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle

_CURAND_PHILOX = 161  # CURAND_RNG_PSEUDO_PHILOX4_32_10


def _curand():
    for p in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(p)
        except OSError:
            continue
    return None


def _curand_words(L, seed: int, offset_words: int, n: int) -> np.ndarray:
    gen = ctypes.c_void_p()
    assert L.curandCreateGeneratorHost(ctypes.byref(gen), _CURAND_PHILOX) == 0
    try:
        assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert L.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset_words)) == 0
        out = (ctypes.c_uint32 * n)()
        assert L.curandGenerate(gen, out, ctypes.c_size_t(n)) == 0
        return np.frombuffer(out, dtype=np.uint32).copy()
    finally:
        L.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEF, 0x123456789ABCDEF0, (1 << 64) - 1])
@pytest.mark.parametrize("block", [0, 1, 7, 65535, 65536 * 3 + 7, (1 << 48) + 65536 * 2 + 9,
                                   ((1 << 32) + 5) * 65536 + 11])
def test_philox_matches_curand_host_generator(seed, block):
    L = _curand()
    if L is None:
        pytest.skip("libcurand not present")
    ref = _curand_words(L, seed, 4 * block, 8)
    k = [seed & 0xFFFFFFFF, seed >> 32]
    for j in range(2):
        b = block + j
        q = b >> 16
        got = oracle.philox4x32_10([q & 0xFFFFFFFF, q >> 32, b & 0xFFFF, 0], k)
        assert np.array_equal(got, ref[4 * j:4 * j + 4]), (hex(seed), b)


def test_philox_upper_counter_words_change_output():
    k = [5, 6]
    base = oracle.philox4x32_10([1, 0, 0, 0], k)
    assert not np.array_equal(base, oracle.philox4x32_10([1, 0, 1, 0], k))
    assert not np.array_equal(base, oracle.philox4x32_10([1, 0, 0, 1], k))
    assert not np.array_equal(oracle.philox4x32_10([1, 0, 1, 0], k), oracle.philox4x32_10([1, 0, 0, 1], k))


def test_sr_uniform_layout():
    # element i uses word (i mod 8) / 2 of counter i / 8; low half for even i
    seed, off = 0xABCDEF0123, 77
    for i in [0, 1, 2, 7, 8, 9, 1000003]:
        g = i // 8
        w = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, off & 0xFFFFFFFF, off >> 32],
                                 [seed & 0xFFFFFFFF, seed >> 32])[(i % 8) // 2]
        expect = int(w) & 0xFFFF if i % 2 == 0 else int(w) >> 16
        assert oracle.sr_uniform16(seed, off, i) == expect


def test_sr_uniform16_is_uniform():
    u = np.array([oracle.sr_uniform16(3, 0, i) for i in range(1 << 16)])
    hist = np.bincount(u >> 12, minlength=16)
    exp = u.size / 16
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 45.0  # 15 dof, p ~ 1e-4


def test_sr_unbiased_inside_range():
    # For values spread over every bin, the mean decoded value over many draws
    # matches the input within 5 sigma, and P(up) matches p.
    xs = [0.1, 0.3, 0.6, 0.9, 1.2, 1.3, 1.7, 2.2, 2.9, 3.3, 3.9, 4.5, 5.5, 5.99]
    n = 1 << 14
    for x in xs:
        codes = np.array([oracle.e2m1_sr(x, oracle.sr_uniform16(99, 5, i)) for i in range(n)])
        vals = np.array([oracle.e2m1_value(int(c)) for c in codes])
        lo = max(m for m in [0, 0.5, 1, 1.5, 2, 3, 4, 6] if m <= x)
        hi = min(m for m in [0, 0.5, 1, 1.5, 2, 3, 4, 6] if m > x)
        p = (x - lo) / (hi - lo)
        sigma = (hi - lo) * np.sqrt(p * (1 - p) / n)
        assert abs(vals.mean() - x) < 5 * sigma + 1e-12, x
        assert set(np.unique(vals)) <= {lo, hi}


def test_sr_streams_depend_on_seed_and_offset_only():
    from synthetic import normal_bf16
    x = normal_bf16((32, 64), 1.0, 4, 1)
    a = oracle.quantize(x, "mx", "row", sr=True, seed=1, offset=2)
    b = oracle.quantize(x, "mx", "row", sr=True, seed=1, offset=2)
    c = oracle.quantize(x, "mx", "row", sr=True, seed=1, offset=3)
    d = oracle.quantize(x, "mx", "row", sr=True, seed=2, offset=2)
    assert np.array_equal(a["codes"], b["codes"])
    assert not np.array_equal(a["codes"], c["codes"])
    assert not np.array_equal(a["codes"], d["codes"])
    # scales never depend on SR (Sec. 2.5: scale values remain deterministic)
    r = oracle.quantize(x, "mx", "row")
    assert np.array_equal(a["scales"], r["scales"])
