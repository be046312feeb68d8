"""Pins of the oracle's QKV producer with RoPE (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 3.2: the Q/K projection applies RoPE and the required
layout; the backward turns the gradients back and restores the QKV layout).
Readings: rotate-half pairs (i, i + D/2), angle p * theta^(-2i/D) with
theta = 500000, position p = token mod S, head-major outputs [heads][T][D]."""
import numpy as np

import oracle
from synthetic import bf16_bits_from_f32, normal_bf16

D = 128


def test_tables_are_the_angles():
    S = 64
    c, s = oracle.rope_tables(S, D)
    assert np.array_equal(c[0], np.ones(D // 2, np.float32)) and np.array_equal(s[0], np.zeros(D // 2, np.float32))
    p = np.arange(S)[:, None].astype(np.float64)
    ang = p * oracle.ROPE_THETA ** (-2.0 * np.arange(D // 2)[None, :] / D)
    assert np.array_equal(c, np.cos(ang).astype(np.float32))
    assert np.array_equal(s, np.sin(ang).astype(np.float32))


def _complex_rotation(x_bits, c, s, inverse=False):
    """Independent binary64 statement of the rotation: z = x_lo + i x_hi
    turned by e^(+-i phi)."""
    x = oracle.bf16_to_f32(x_bits).astype(np.float64)
    z = x[..., :D // 2] + 1j * x[..., D // 2:]
    e = (c.astype(np.float64) + 1j * s.astype(np.float64))
    w = z * (np.conj(e) if inverse else e)
    return np.concatenate([w.real, w.imag], axis=-1)


def test_forward_layout_and_rotation():
    T, S, hq, hkv = 192, 64, 4, 2
    qkv = normal_bf16((T, (hq + 2 * hkv) * D), 1.0, 81, 1)
    c, s = oracle.rope_tables(S, D)
    q, k, v = oracle.qkv_rope_fwd(qkv, S, hq, hkv, c, s)
    assert q.shape == (hq, T, D) and k.shape == (hkv, T, D) and v.shape == (hkv, T, D)
    pos = np.arange(T) % S
    for h in range(hkv):  # V heads are copied, head-major
        assert np.array_equal(v[h], qkv[:, (hq + hkv + h) * D:(hq + hkv + h + 1) * D])
    for h, (out, col) in enumerate([(q[i], i) for i in range(hq)] + [(k[i], hq + i) for i in range(hkv)]):
        src = qkv[:, col * D:(col + 1) * D]
        ref = _complex_rotation(src, c[pos], s[pos])
        got = oracle.bf16_to_f32(out).astype(np.float64)
        # binary32 products and sums, then one bf16 rounding
        bound = np.abs(ref) * 2.0 ** -8 + 4 * 2.0 ** -24 * np.abs(oracle.bf16_to_f32(src)).max(axis=1, keepdims=True)
        assert (np.abs(got - ref) <= bound).all(), h


def test_backward_is_the_transposed_rotation():
    T, S, hq, hkv = 128, 32, 2, 1
    c, s = oracle.rope_tables(S, D)
    dq = normal_bf16((hq, T, D), 1.0, 82, 1)
    dk = normal_bf16((hkv, T, D), 1.0, 82, 2)
    dv = normal_bf16((hkv, T, D), 1.0, 82, 3)
    dqkv = oracle.qkv_rope_bwd(dq, dk, dv, S, c, s)
    pos = np.arange(T) % S
    assert np.array_equal(dqkv[:, (hq + hkv) * D:], dv[0])
    for h in range(hq):
        ref = _complex_rotation(dq[h], c[pos], s[pos], inverse=True)
        got = oracle.bf16_to_f32(dqkv[:, h * D:(h + 1) * D]).astype(np.float64)
        assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 4 * 2.0 ** -24 * 8).all()


def test_rotation_is_orthogonal_and_relative():
    # in exact arithmetic the turned dot product depends only on p - p'
    S = 256
    c, s = oracle.rope_tables(S, D)
    rng = np.random.default_rng(3)
    qv, kv = rng.standard_normal(D), rng.standard_normal(D)

    def turn(x, p):
        z = (x[:D // 2] + 1j * x[D // 2:]) * (c[p].astype(np.float64) + 1j * s[p].astype(np.float64))
        return np.concatenate([z.real, z.imag])

    for p, pp in ((5, 3), (100, 37), (200, 199)):
        a = turn(qv, p) @ turn(kv, pp)
        b = turn(qv, p - pp) @ turn(kv, 0)
        assert abs(a - b) <= 1e-5 * np.abs(qv).sum() * np.abs(kv).max()
        assert abs(np.linalg.norm(turn(qv, p)) - np.linalg.norm(qv)) <= 1e-6 * np.linalg.norm(qv)


def test_forward_then_backward_returns_the_input():
    T, S, hq, hkv = 64, 64, 2, 1
    c, s = oracle.rope_tables(S, D)
    x = bf16_bits_from_f32((np.random.default_rng(4).integers(-8, 8, (T, (hq + 2 * hkv) * D)) / 4.0).astype(np.float32))
    q, k, v = oracle.qkv_rope_fwd(x, S, hq, hkv, c, s)
    back = oracle.qkv_rope_bwd(q, k, v, S, c, s)
    # two bf16 roundings: within a few ulps of the input
    xf, bf = oracle.bf16_to_f32(x).astype(np.float64), oracle.bf16_to_f32(back).astype(np.float64)
    assert (np.abs(bf - xf) <= 2.0 ** -6 * np.abs(xf).max() + 1e-30).all()
    assert np.array_equal(back[:, (hq + hkv) * D:], x[:, (hq + hkv) * D:])
