"""Brute-force pins of the oracle's block encoders (Format-Aware Fusion for
Fast FP4 Pretraining, Sec. 2.2 Eq. 1, Sec. 2.2.1, Sec. 2.2.2, Sec. 2.4, Sec.
2.5 Eq. 9).

Every expected value here comes from enumeration in exact rational
arithmetic, not from the oracle's own formulas: for a block, every candidate
scale (all 255 E8M0 exponents, all 127 finite E4M3 scales) and every one of
the 16 E2M1 codes is tried, and the choice the format definition fixes is
taken (the smallest scale that does not clip; the nearest code, ties to the
even code).  Inputs are seeded random blocks plus adversarial ones: exact
rounding ties, amax exactly on and just past a scale boundary, zeros and
negative zeros, bf16 subnormals, values near the bf16 maximum, lone outliers.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from synthetic import bf16_bits_from_f32, f32_from_bf16_bits

MAG = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
RATIO_087 = Fraction(87, 100)  # the pages' adaptive 2D32 threshold a/s < 0.87


def _frac(x) -> Fraction:
    return Fraction(float(x))


def _signbit(x_bits: int) -> int:
    return 8 if x_bits & 0x8000 else 0


def nearest_code(v: Fraction, sign: int) -> int:
    """Argmin over the 8 magnitudes of |v| - q (ties to the even index), with
    the input's sign bit; beyond 6 the nearest magnitude is 6 (saturation)."""
    a = abs(v)
    best, bestd = None, None
    for k, q in enumerate(MAG):
        d = abs(a - q)
        if bestd is None or d < bestd or (d == bestd and k % 2 == 0):
            best, bestd = k, d
    return sign | best


def mx_min_exponent(amax: Fraction) -> int:
    """The smallest E8M0 exponent e in [-127, 127] with 6 * 2^e >= amax,
    found by trying every exponent in order."""
    for e in range(-127, 128):
        if Fraction(6) * Fraction(2) ** e >= amax:
            return e
    return 127


def e4m3_values():
    """All finite non-negative E4M3 values by code (OCP: bias 7, 3 fraction
    bits, exponent field 0 subnormal, 0x7F NaN)."""
    out = []
    for c in range(0x7F):
        E, m = c >> 3, c & 7
        out.append(Fraction(m, 8) * Fraction(2) ** -6 if E == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (E - 7))
    return out


E4M3 = e4m3_values()


def e4m3_nearest(s: Fraction) -> int:
    """Nearest E4M3 code to s >= 0 by enumeration (ties to the even code);
    values past the largest finite one saturate to it."""
    best, bestd = None, None
    for c, q in enumerate(E4M3):
        d = abs(s - q)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best


def _bf16(vals) -> np.ndarray:
    return bf16_bits_from_f32(np.asarray(vals, np.float32))


def _mx_blocks(n_random: int, seed: int) -> np.ndarray:
    """(N, 32) bf16 blocks: random magnitudes over a wide range plus
    adversarial constructions."""
    rng = np.random.default_rng(seed)
    blocks = []
    for _ in range(n_random):
        e = rng.integers(-130, 118)
        v = rng.standard_normal(32) * 2.0 ** float(e)
        if rng.random() < 0.3:
            v[rng.integers(0, 32)] *= 20.0  # a lone outlier
        if rng.random() < 0.2:
            v[rng.integers(0, 32, 8)] = 0.0
        blocks.append(_bf16(v))
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for e in (-20, -1, 0, 3, 40):
        s = 2.0 ** e
        # every rounding tie of the grid, both signs, with amax exactly 6 * 2^e
        v = [t * s for t in ties] + [-t * s for t in ties] + [6.0 * s] + [0.1 * s] * 17
        blocks.append(_bf16(v))
        # amax just past 6 * 2^e (the next bf16 value): the exponent moves up
        nxt = float(f32_from_bf16_bits(np.array([_bf16([6.0 * s])[0] + 1], np.uint16))[0])
        blocks.append(_bf16([nxt] + [t * s for t in ties] * 4 + [-t * s for t in ties][:3]))
        # amax exactly 3 * 2^e (a power-of-two boundary of the ratio)
        blocks.append(_bf16([3.0 * s] + [0.3 * s] * 31))
    # zeros, negative zeros, one nonzero, bf16 subnormals, the bf16 maximum
    blocks.append(np.zeros(32, np.uint16))
    blocks.append(np.full(32, 0x8000, np.uint16))
    z = np.full(32, 0x8000, np.uint16)
    z[5] = _bf16([1e-3])[0]
    blocks.append(z)
    blocks.append(np.arange(1, 33, dtype=np.uint16))          # positive bf16 subnormals
    blocks.append((np.arange(1, 33) | 0x8000).astype(np.uint16))
    blocks.append(np.full(32, 0x7F7F, np.uint16))              # largest finite bf16
    blocks.append(_bf16(np.linspace(-3.0e38, 3.0e38, 32)))
    return np.stack(blocks).astype(np.uint16)


def test_mx_blocks_brute_force():
    x = _mx_blocks(1200, 11)
    q = oracle.quantize(x, "mx", "row")
    xf = f32_from_bf16_bits(x)
    for b in range(x.shape[0]):
        vals = [_frac(t) for t in xf[b]]
        amax = max(abs(t) for t in vals)
        e = mx_min_exponent(amax)
        assert int(q["scales"][b, 0]) == e + 127, f"block {b}: scale"
        scale = Fraction(2) ** e
        for j in range(32):
            want = nearest_code(vals[j] / scale, _signbit(int(x[b, j])))
            assert int(q["codes"][b, j]) == want, f"block {b} element {j}"


def test_mx_weight2d_tiles_brute_force():
    """32x32 weight tiles: the exponent is the smallest non-clipping one, or
    one finer when the tile amax is below 0.87 of that span (Sec. 2.2.1); the
    codes are the nearest grid values of the tile-scaled weights, saturating."""
    rng = np.random.default_rng(5)
    tiles = []
    # tile amax ratios a / (6 * 2^e) swept across 0.87 on bf16 values
    for a in list(np.linspace(3.05, 6.0, 40)) + [5.21875, 5.25, 5.1875, 3.0, 6.0]:
        t = rng.standard_normal((32, 32)) * 0.3
        t = np.clip(t, -a * 0.9, a * 0.9)
        t[rng.integers(0, 32), rng.integers(0, 32)] = a * (1 if rng.random() < 0.5 else -1)
        tiles.append(t * 2.0 ** float(rng.integers(-30, 30)))
    tiles.append(np.zeros((32, 32)))
    x = _bf16(np.concatenate(tiles, axis=1))  # (32, 32 * tiles)
    q = oracle.quantize(x, "mx", "row", weight2d=True)
    xf = f32_from_bf16_bits(x)
    fine_seen = coarse_seen = 0
    for t in range(x.shape[1] // 32):
        vals = [[_frac(v) for v in row[32 * t:32 * t + 32]] for row in xf]
        amax = max(abs(v) for row in vals for v in row)
        e = mx_min_exponent(amax)
        if amax > 0 and amax / (6 * Fraction(2) ** e) < RATIO_087 and e > -127:
            e -= 1
            fine_seen += 1
        else:
            coarse_seen += 1
        assert all(int(q["scales"][r, t]) == e + 127 for r in range(32)), f"tile {t}: scale"
        scale = Fraction(2) ** e
        for r in range(32):
            for j in range(32):
                want = nearest_code(vals[r][j] / scale, _signbit(int(x[r, 32 * t + j])))
                assert int(q["codes"][r, 32 * t + j]) == want, f"tile {t} ({r}, {j})"
    assert fine_seen > 5 and coarse_seen > 5


def _f32(v) -> np.float32:
    return np.float32(v)


def _nv_expect_block(vals_f32, x_bits, senc: np.float32):
    """The global-NVFP4 encoding of one 16-value block under the outer factor
    senc (the stated binary32 operation order: s_raw = fl32(fl32(a / 6) * S_enc),
    m = fl32(S_enc / delta), v = fl32(x * m)), with the E4M3 scale and the
    E2M1 codes found by enumeration."""
    a = max(abs(_f32(v)) for v in vals_f32)
    s_raw = _f32(_f32(a / _f32(6.0)) * senc)
    d = e4m3_nearest(_frac(s_raw))
    dv = E4M3[d]
    m = _f32(0.0) if d == 0 else _f32(senc / _f32(float(dv)))
    codes = [nearest_code(_frac(_f32(_f32(v) * m)), _signbit(int(xb))) for v, xb in zip(vals_f32, x_bits)]
    return d, codes


def _nv_rows(n_rows: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n_rows):
        v = rng.standard_normal(64) * np.exp(rng.uniform(-12, 3, 64).repeat(1))
        v[rng.integers(0, 64, 4)] = 0.0
        rows.append(v)
    x = np.array(rows)
    x[0, 0] = 37.0  # tensor amax
    return _bf16(x)


def test_nv_global_blocks_brute_force():
    x = _nv_rows(300, 17)
    # blocks whose scale lands on E4M3 rounding ties and on the saturation edge
    senc = _f32(np.float32(2688.0) / np.float32(37.0))
    extra = []
    for t in (E4M3[10] + E4M3[11]) / 2, (E4M3[40] + E4M3[41]) / 2, Fraction(448), Fraction(1, 2048):
        a = float(t) * 6.0 / float(senc)
        extra.append(np.concatenate([[a], np.linspace(-a, a, 15), np.zeros(48)]))
    x = np.concatenate([x, _bf16(np.array(extra))])
    q = oracle.quantize(x, "nv_global", "row")
    xf = f32_from_bf16_bits(x)
    A = max(abs(_f32(v)) for v in xf.ravel())
    S = _f32(np.float32(2688.0) / A)
    assert q["senc"][0] == S
    zero_scales = 0
    for r in range(x.shape[0]):
        for b in range(4):
            d, codes = _nv_expect_block(xf[r, 16 * b:16 * b + 16], x[r, 16 * b:16 * b + 16], S)
            assert int(q["scales"][r, b]) == d, f"row {r} block {b}: scale"
            assert [int(c) for c in q["codes"][r, 16 * b:16 * b + 16]] == codes, f"row {r} block {b}"
            zero_scales += d == 0
    assert zero_scales > 0  # some blocks vanish under the tensor factor (Sec. 2.2.2)


def test_nv_weight2d_tiles_brute_force():
    rng = np.random.default_rng(23)
    w = rng.standard_normal((32, 64)) * 0.02
    w[rng.integers(0, 32, 10), rng.integers(0, 64, 10)] *= 30
    w[16:32, 0:16] *= 1e-4
    x = _bf16(w)
    q = oracle.quantize(x, "nv_local", "row", weight2d=True)
    xf = f32_from_bf16_bits(x)
    A = max(abs(_f32(v)) for v in xf.ravel())
    S = _f32(np.float32(2688.0) / A)
    assert (q["senc"] == S).all()
    for tr in range(2):
        for tc in range(4):
            tile = xf[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16]
            a = max(abs(_f32(v)) for v in tile.ravel())
            d = e4m3_nearest(_frac(_f32(_f32(a / _f32(6.0)) * S)))
            m = _f32(0.0) if d == 0 else _f32(S / _f32(float(E4M3[d])))
            for r in range(16):
                assert int(q["scales"][16 * tr + r, tc]) == d
                for j in range(16):
                    c = int(q["codes"][16 * tr + r, 16 * tc + j])
                    want = nearest_code(_frac(_f32(_f32(tile[r, j]) * m)), _signbit(int(x[16 * tr + r, 16 * tc + j])))
                    assert c == want


def test_nv_decode_error_bound_per_element():
    """|x - x_hat| <= (half a grid step at |v| + the saturation excess past 6
    + two binary32 roundings) * delta / S_enc, where v = x * S_enc / delta is
    the exactly scaled value; and delta is within E4M3 rounding of
    amax * S_enc / 6 (relative 2^-4 for normal scales, 2^-10 absolute below)."""
    x = _nv_rows(200, 29)
    q = oracle.quantize(x, "nv_global", "row")
    xf = f32_from_bf16_bits(x).astype(np.float64)
    xh = oracle.dequantize(q)
    S = float(q["senc"][0])
    for r in range(x.shape[0]):
        for b in range(4):
            blk = xf[r, 16 * b:16 * b + 16]
            d = int(q["scales"][r, b])
            dv = float(E4M3[d])
            target = np.abs(blk).max() * S / 6.0
            if d == 0:
                assert target < 2.0 ** -10 * (1 + 2.0 ** -20)
                assert (xh[r, 16 * b:16 * b + 16] == 0).all()
                continue
            tol_rel = 2.0 ** -4 if dv >= 2.0 ** -6 else 0.0
            assert abs(dv - target) <= max(tol_rel * target, 2.0 ** -10) * (1 + 2.0 ** -20) or dv == 448.0
            v = np.abs(blk) * S / dv
            half = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
            bound = (half + np.maximum(0.0, v - 6.0) + v * 2.0 ** -22) * dv / S
            err = np.abs(blk - xh[r, 16 * b:16 * b + 16])
            assert (err <= bound * (1 + 1e-12)).all(), (r, b)


def _threshold_code(a: float) -> int:
    """E2M1 magnitude index of a >= 0 by the midpoints between neighbours
    (a midpoint goes to the neighbour with an even index)."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for k in range(7):
        mid = (mags[k] + mags[k + 1]) / 2
        if a < mid or (a == mid and k % 2 == 0):
            return k
    return 7


def test_e2m1_rn_all_bf16_times_every_landing_exponent():
    """Every finite bf16 value times every power of two 2^-e (e an E8M0
    exponent) that lands its magnitude in [2^-4, 8], plus one landing below:
    the oracle's RN code equals the threshold rule (ties to even)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = f32_from_bf16_bits(bits).astype(np.float64)
    fin = np.isfinite(f) & (f != 0)
    checked = 0
    for b, v in zip(bits[fin], f[fin]):
        k = math.floor(math.log2(abs(v)))
        sign = 8 if b & 0x8000 else 0
        for e in range(k - 3, k + 6):
            if not -127 <= e <= 127:
                continue
            s = v * 2.0 ** -e  # exact: a bf16 value times a power of two
            if abs(s) > 8:
                continue
            assert oracle.e2m1_rn(s) == sign | _threshold_code(abs(s)), (hex(int(b)), e)
            checked += 1
    assert checked > 400000
    # zeros keep their sign bit
    assert oracle.e2m1_rn(0.0) == 0 and oracle.e2m1_rn(-0.0) == 8


@pytest.mark.parametrize("x", [0.1, 0.3, 0.6, 0.9, 1.2, 1.3, 1.7, 2.2, 2.9, 3.3, 3.9, 4.5, 5.5, 5.96875])
def test_sr_up_probability_at_2_22_draws(x):
    """Sec. 2.5 (Eq. 9): with a 16-bit uniform u, the value rounds up iff
    u / 2^16 < p, so the exact probability of rounding up is
    ceil(p 2^16) / 2^16, within 2^-16 of p.  2^22 draws through the tensor
    path (one block scale of 1 per row, consecutive logical indices): the
    observed fraction is within 5 sigma of it, and the draws only ever take
    the two neighbouring grid values."""
    xb = _bf16([x])[0]
    xv = Fraction(float(f32_from_bf16_bits(np.array([xb], np.uint16))[0]))
    lo = max(k for k in range(8) if MAG[k] <= xv)
    p = (xv - MAG[lo]) / (MAG[lo + 1] - MAG[lo])
    p_up = Fraction(math.ceil(p * 65536), 65536)
    assert abs(p_up - p) <= Fraction(1, 65536)
    rows = (1 << 22) // 31 + 1
    t = np.full((rows, 32), xb, np.uint16)
    t[:, 0] = _bf16([6.0])[0]  # block amax 6: exponent 0, the value is its own scaled value
    q = oracle.quantize(t, "mx", "row", sr=True, seed=12345, offset=7)
    assert (q["scales"] == 127).all()
    c = q["codes"][:, 1:].ravel()
    assert set(np.unique(c).tolist()) <= {lo, lo + 1}
    n = c.size
    up = int((c == lo + 1).sum())
    pf = float(p_up)
    sigma = math.sqrt(pf * (1 - pf) / n)
    assert abs(up / n - pf) <= 5 * sigma + 1e-12, (x, up / n, pf)
