"""Pins of the oracle's tensor quantizers (Format-Aware Fusion for Fast FP4
Pretraining, Sec. 2.2-2.4): decode-error bounds, the transposition invariant
of 2D weight encodings (Eq. 8), and the relations between global and CTA-local
NVFP4 outer factors."""
import numpy as np
import pytest

import oracle
from synthetic import f32_from_bf16_bits, normal_bf16, with_outliers_bf16, bf16_bits_from_f32

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _half_step(v):
    """Half the E2M1 grid spacing around |v| (v already on the code scale)."""
    a = np.abs(v)
    return np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))


def test_mx_row_decode_error_bound_and_block_sizes(paper_facts):
    x = with_outliers_bf16((64, 256), 1.0, 1e-2, 20.0, 5, 1)
    q = oracle.quantize(x, "mx", "row")
    assert q["bs"] == paper_facts["mx_block"]
    xf = f32_from_bf16_bits(x).astype(np.float64)
    xh = oracle.dequantize(q)
    step = 2.0 ** (q["scales"].astype(np.int64) - 127)
    step = np.repeat(step, 32, axis=1)
    # upward scales never clip: |x| <= 6 * 2^e, error <= half a grid step
    assert (np.abs(xf) <= 6 * step).all()
    assert (np.abs(xf - xh) <= _half_step(xf / step) * step).all()


def test_mx_col_view_is_row_view_of_transpose():
    x = normal_bf16((96, 128), 1.0, 6, 1)
    c = oracle.quantize(x, "mx", "col")
    r = oracle.quantize(np.ascontiguousarray(x.T), "mx", "row")
    assert np.array_equal(c["codes"], r["codes"]) and np.array_equal(c["scales"], r["scales"])


@pytest.mark.parametrize("route", ["mx", "nv_global", "nv_local"])
def test_weight2d_transposition_invariant(route):
    w = normal_bf16((128, 256), 0.02, 7, 2)
    r = oracle.quantize(w, route, "row", weight2d=True)
    c = oracle.quantize(w, route, "col", weight2d=True)
    # Eq. 8: the two views decode to the same weight, element for element
    assert np.array_equal(oracle.dequantize(r), oracle.dequantize(c).T)
    assert np.array_equal(r["codes"], c["codes"].T)


def test_mx_weight2d_uses_fine_scale_and_bounded_clip():
    # one 32x32 tile whose amax ratio is below 0.87 takes e-1 and may clip at 6
    w = np.full((32, 32), 1.0, np.float32)
    w[0, 0] = 4.0  # ratio 4/6 < 0.87 -> finer exponent
    q = oracle.quantize(bf16_bits_from_f32(w), "mx", "row", weight2d=True)
    e = int(q["scales"][0, 0]) - 127
    assert e == oracle.e8m0_exponent_up(4.0) - 1
    w[0, 0] = 5.5  # ratio 5.5/6 >= 0.87 -> upward exponent
    q = oracle.quantize(bf16_bits_from_f32(w), "mx", "row", weight2d=True)
    assert int(q["scales"][0, 0]) - 127 == oracle.e8m0_exponent_up(5.5)


def test_nv_global_bound_and_zero_block(paper_facts):
    x = with_outliers_bf16((32, 128), 1.0, 1e-2, 20.0, 8, 1).copy()
    xf = f32_from_bf16_bits(x)
    # a block far below the tensor amax: its E4M3 scale underflows and it decodes to 0
    tiny = bf16_bits_from_f32(np.full(16, 1e-9, np.float32))
    x[3, 16:32] = tiny
    q = oracle.quantize(x, "nv_global", "row")
    assert q["bs"] == paper_facts["nv_block"]
    xh = oracle.dequantize(q)
    A = float(np.abs(f32_from_bf16_bits(x)).max())
    assert np.abs(xh).max() <= A * (1 + 2.0 ** -3)
    assert q["scales"][3, 1] == 0 and (xh[3, 16:32] == 0).all()


def test_nv_scale_one_block_is_plain_e2m1():
    # tensor amax 2688 -> S_enc = 1; a block with amax 6 -> delta = 1.0, m = 1
    v = np.linspace(-6, 6, 16).astype(np.float32)
    x = np.zeros((1, 32), np.float32)
    x[0, :16] = v
    x[0, 16] = 2688.0
    xb = bf16_bits_from_f32(x)
    q = oracle.quantize(xb, "nv_global", "row")
    assert q["senc"][0] == 1.0 and q["scales"][0, 0] == 0x38
    vb = f32_from_bf16_bits(xb[0, :16])
    assert list(q["codes"][0, :16]) == [oracle.e2m1_rn(float(t)) for t in vb]


def test_nv_local_equals_global_when_strips_share_amax():
    x = normal_bf16((256, 256), 1.0, 9, 1).copy()
    big = bf16_bits_from_f32(np.array([7.0], np.float32))[0]
    for s in range(0, 256, 128):  # put the same amax in every row strip and column strip
        x[s, s] = big
    for view in ("row", "col"):
        g = oracle.quantize(x, "nv_global", view)
        l = oracle.quantize(x, "nv_local", view)
        assert np.array_equal(g["codes"], l["codes"]) and np.array_equal(g["scales"], l["scales"])
        assert np.array_equal(g["senc"], l["senc"])


def test_nv_local_factors_are_per_strip():
    x = normal_bf16((256, 128), 1.0, 10, 1)
    q = oracle.quantize(x, "nv_local", "row")
    xf = f32_from_bf16_bits(x)
    for s in (0, 128):
        assert (q["senc"][s:s + 128] == oracle.nv_senc(float(np.abs(xf[s:s + 128]).max()))).all()
    qc = oracle.quantize(x, "nv_local", "col")
    assert (qc["senc"] == oracle.nv_senc(float(np.abs(xf).max()))).all()


def test_nv_weight2d_local_factor_is_tensor_amax():
    w = normal_bf16((64, 64), 0.02, 11, 1)
    a = oracle.quantize(w, "nv_local", "row", weight2d=True)
    b = oracle.quantize(w, "nv_global", "row", weight2d=True)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["senc"], b["senc"])


def test_sr_only_on_row_view_and_hadamard_only_on_mx_col():
    x = normal_bf16((32, 64), 1.0, 12, 1)
    with pytest.raises(ValueError):
        oracle.quantize(x, "mx", "col", sr=True)
    with pytest.raises(ValueError):
        oracle.quantize(x, "mx", "row", hadamard=True, signs=np.ones(16, np.int8))


def test_hadamard_col_view_preserves_dot_before_quantization():
    from synthetic import hadamard_signs
    x = normal_bf16((64, 32), 1.0, 13, 1)
    dy = normal_bf16((64, 16), 1.0, 13, 2)
    s = hadamard_signs(13)
    qx = oracle.quantize(x, "mx", "col", hadamard=True, signs=s)
    qd = oracle.quantize(dy, "mx", "col", hadamard=True, signs=s)
    # the transformed-and-quantized Wgrad approximates dY^T X (the transform cancels)
    ref = f32_from_bf16_bits(dy).astype(np.float64).T @ f32_from_bf16_bits(x).astype(np.float64)
    got = oracle.gemm(qd, qx)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.2


def test_sr_of_a_block_uses_the_whole_tensors_indices():
    """Stochastic rounding draws its counter from the element's logical index
    in the whole tensor (Sec. 2.5): a block quantized with its origin in the
    larger tensor reproduces that block of the whole-tensor result, and the
    same block quantized as a tensor of its own does not."""
    x = normal_bf16((256, 512), 1.0, 61, 1)
    r0, c0 = 128, 256
    blk = np.ascontiguousarray(x[r0:r0 + 128, c0:c0 + 128])
    whole = oracle.quantize(x, "mx", "row", sr=True, seed=5, offset=2)
    part = oracle.quantize(blk, "mx", "row", sr=True, seed=5, offset=2, sr_origin=(r0, c0), sr_cols=512)
    assert np.array_equal(part["codes"], whole["codes"][r0:r0 + 128, c0:c0 + 128])
    alone = oracle.quantize(blk, "mx", "row", sr=True, seed=5, offset=2)
    assert not np.array_equal(alone["codes"], part["codes"])
    # CTA-local NVFP4: a 128-row strip carries its own factor, so a strip
    # quantized with its origin equals the whole tensor's rows
    whole = oracle.quantize(x, "nv_local", "row", sr=True, seed=5, offset=2)
    strip = oracle.quantize(np.ascontiguousarray(x[r0:r0 + 128]), "nv_local", "row", sr=True, seed=5, offset=2,
                            sr_origin=(r0, 0), sr_cols=512)
    assert np.array_equal(strip["codes"], whole["codes"][r0:r0 + 128])
    assert np.array_equal(strip["scales"], whole["scales"][r0:r0 + 128])
