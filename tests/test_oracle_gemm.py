"""Pins of the oracle contraction (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 2.3 Eqs. 4-6): exact integer special cases and agreement
with numpy's matmul over the decoded operands."""
import numpy as np

import oracle
from synthetic import normal_bf16


def test_unit_scale_codes_give_exact_integer_gemm():
    rng = np.random.default_rng(0)
    M, N, K = 64, 48, 128
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    for fmt, bs, one in ((0, 32, 127), (1, 16, 0x38)):
        a = dict(codes=ca, scales=np.full((M, K // bs), one, np.uint8), senc=None, fmt=fmt, bs=bs)
        b = dict(codes=cb, scales=np.full((N, K // bs), one, np.uint8), senc=None, fmt=fmt, bs=bs)
        ia = np.vectorize(lambda c: int(round(2 * oracle.e2m1_value(int(c)))))(ca).astype(np.int64)
        ib = np.vectorize(lambda c: int(round(2 * oracle.e2m1_value(int(c)))))(cb).astype(np.int64)
        want = (ia @ ib.T).astype(np.float64) / 4.0
        assert np.array_equal(oracle.gemm(a, b), want)


def test_gemm_matches_numpy_on_decoded_and_sampled_matches_full():
    x = normal_bf16((128, 256), 1.0, 1, 1)
    w = normal_bf16((64, 256), 0.02, 1, 2)
    for route in ("mx", "nv_global", "nv_local"):
        a = oracle.quantize(x, route, "row")
        b = oracle.quantize(w, route, "row", weight2d=True)
        full = oracle.gemm(a, b)
        ref = oracle.dequantize(a) @ oracle.dequantize(b).T
        assert np.allclose(full, ref, rtol=1e-12, atol=1e-300)
        ms = np.array([0, 5, 127, 64])
        ns = np.array([0, 63, 1, 32])
        s, sa = oracle.gemm_sampled(a, b, ms, ns)
        assert np.allclose(s, full[ms, ns], rtol=1e-12)
        assert (sa >= np.abs(s)).all()
