"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (same entry points, flags, seeds and output buffers):

  MXFP4 Llama-3-8B W1 linear  X 8192x4096, W 14336x4096, dY 8192x14336 with
                              SR on the row-facing dY and fixed-sign H32 on
                              the column-facing X and dY;
  NVFP4 attention projections X 8192x4096, W 4096x4096 and 6144x4096, global
                              and CTA-local, 2D16 weights, SR on dY;
  fused SwiGLU FFN            T 16384, d 4096, f 14336;
  32-block 27/5 hybrid stack  T 8192.

(Format-Aware Fusion for Fast FP4 Pretraining, Secs. 2.2-2.5, 3.2, 3.3.)
Every code and scale byte of the quantizers is compared with the oracle's.
The contractions are checked on every element of 8 random 128 x 128 output
tiles plus 65,536 random elements, each an FP64 dot product of the oracle's
own operand views (which the GPU's equal bit for bit), against the
tolerance: relative Frobenius error over the sample <= 1e-5 and, per
element, |err| <= 2^-18 * sum_k |a_k b_k|.  The fused producers are checked
on sampled tiles with the masked comparison of masked.py."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack
from masked import assert_view_masked, oriented
from masked import host_view as mhost
from synthetic import config_tensors, normal_bf16
from parity_stats import record

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5
PER_ELEM = 2.0 ** -18


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def same_view(v: F.QView, want: dict, what: str):
    got = mhost(v)
    nc = int(np.sum(got["codes"] != want["codes"]))
    ns = int(np.sum(got["scales"] != want["scales"]))
    assert nc == 0 and ns == 0, f"{what}: {nc} code and {ns} scale mismatches"
    if want["senc"] is not None:
        assert np.array_equal(got["senc"], want["senc"]), f"{what}: outer factors"


def sample_points(M, N, rng, tiles=8, rand=65536):
    ms, ns = [], []
    for _ in range(tiles):
        m0 = int(rng.integers(0, M // 128)) * 128
        n0 = int(rng.integers(0, N // 128)) * 128
        mm, nn = np.meshgrid(np.arange(m0, m0 + 128), np.arange(n0, n0 + 128), indexing="ij")
        ms.append(mm.ravel())
        ns.append(nn.ravel())
    ms.append(rng.integers(0, M, rand))
    ns.append(rng.integers(0, N, rand))
    return np.concatenate(ms).astype(np.int64), np.concatenate(ns).astype(np.int64)


def check_sampled(out: torch.Tensor, a: dict, b: dict, what: str, rng):
    M, N = out.shape
    ms, ns = sample_points(M, N, rng)
    got = out[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].float().cpu().numpy().astype(np.float64)
    ref, absref = oracle.gemm_sampled(a, b, ms, ns)
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    err = np.abs(got - ref)
    ratio = (err / np.maximum(absref, 1e-300)).max()
    record(what, fro=fro, err_over_sum_abs=ratio)
    assert fro <= REL_FRO, f"{what}: relative Frobenius {fro:.3e} over the sample"
    assert (err <= PER_ELEM * absref + 1e-30).all(), f"{what}: max err / sum|ab| = {ratio:.3e}"


# ------------------------------------------------ MXFP4 W1-shaped linear ----
def test_mxfp4_llama3_8b_w1_full():
    T, di, do = 8192, 4096, 14336
    t = config_tensors("c2_mx_w1")
    signs = [int(s) for s in t["signs"]]
    X, W, DY = to_dev(t["x"]), to_dev(t["w"]), to_dev(t["dy"])
    xr, xc = F.alloc_view("mx", T, di), F.alloc_view("mx", di, T)
    wr, wc = F.alloc_view("mx", do, di), F.alloc_view("mx", di, do)
    dr, dc = F.alloc_view("mx", T, do), F.alloc_view("mx", do, T)
    F.fp4_quantize(X, "mx", 3, F.FP4_FLAG_HADAMARD_COL, hadamard_signs=signs, row_out=xr, col_out=xc)
    F.fp4_quantize(W, "mx", 3, F.FP4_FLAG_WEIGHT_2D, row_out=wr, col_out=wc)
    F.fp4_quantize(DY, "mx", 3, F.FP4_FLAG_SR_ROW | F.FP4_FLAG_HADAMARD_COL, sr_seed=1, sr_offset=0,
                   hadamard_signs=signs, row_out=dr, col_out=dc)
    Y = F.fp4_linear_fprop(xr, wr)
    DX = F.fp4_linear_dgrad(dr, wc)
    DW = F.fp4_linear_wgrad(dc, xc)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    del X, W, DY
    ov = dict(xr=oracle.quantize(t["x"], "mx", "row"),
              xc=oracle.quantize(t["x"], "mx", "col", hadamard=True, signs=t["signs"]),
              wr=oracle.quantize(t["w"], "mx", "row", weight2d=True),
              wc=oracle.quantize(t["w"], "mx", "col", weight2d=True),
              dr=oracle.quantize(t["dy"], "mx", "row", sr=True, seed=1, offset=0),
              dc=oracle.quantize(t["dy"], "mx", "col", hadamard=True, signs=t["signs"]))
    for k, v in dict(xr=xr, xc=xc, wr=wr, wc=wc, dr=dr, dc=dc).items():
        same_view(v, ov[k], f"W1 {k}")
    rng = np.random.default_rng(8)
    check_sampled(Y, ov["xr"], ov["wr"], "Fprop", rng)
    check_sampled(DX, ov["dr"], ov["wc"], "Dgrad", rng)
    check_sampled(DW, ov["dc"], ov["xc"], "Wgrad", rng)


# ------------------------------------------- NVFP4 attention projections ----
@pytest.fixture(scope="module")
def attn_tensors():
    return config_tensors("c3_nv_attn")


@pytest.mark.parametrize("route", ["nv_global", "nv_local"])
@pytest.mark.parametrize("wname,dyname", [("w", "dy"), ("w_qkv", "dy_qkv")])
def test_nvfp4_attention_projection_full(attn_tensors, route, wname, dyname):
    t = attn_tensors
    X, Wt, DYt = to_dev(t["x"]), to_dev(t[wname]), to_dev(t[dyname])
    T, n_in = X.shape
    n_out = Wt.shape[0]
    ws = torch.empty(max(F.fp4_quantize_workspace_bytes(route, T, n_out), F.fp4_quantize_workspace_bytes(route, n_out, n_in),
                         16), dtype=torch.uint8, device="cuda")
    xr, xc = F.fp4_quantize(X, route, 3, 0, workspace=ws)
    wr, wc = F.fp4_quantize(Wt, route, 3, F.FP4_FLAG_WEIGHT_2D, workspace=ws)
    dr, dc = F.fp4_quantize(DYt, route, 3, F.FP4_FLAG_SR_ROW, sr_seed=2, workspace=ws)
    Y = F.fp4_linear_fprop(xr, wr)
    DX = F.fp4_linear_dgrad(dr, wc)
    DW = F.fp4_linear_wgrad(dc, xc)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    ov = dict(xr=oracle.quantize(t["x"], route, "row"), xc=oracle.quantize(t["x"], route, "col"),
              wr=oracle.quantize(t[wname], route, "row", weight2d=True),
              wc=oracle.quantize(t[wname], route, "col", weight2d=True),
              dr=oracle.quantize(t[dyname], route, "row", sr=True, seed=2, offset=0),
              dc=oracle.quantize(t[dyname], route, "col"))
    for k, v in dict(xr=xr, xc=xc, wr=wr, wc=wc, dr=dr, dc=dc).items():
        same_view(v, ov[k], f"{route} {wname} {k}")
    rng = np.random.default_rng(9)
    check_sampled(Y, ov["xr"], ov["wr"], f"{route} Fprop", rng)
    check_sampled(DX, ov["dr"], ov["wc"], f"{route} Dgrad", rng)
    check_sampled(DW, ov["dc"], ov["xc"], f"{route} Wgrad", rng)


# ---------------------------------------------------- fused SwiGLU FFN ----
def _bf16_close(got_bits, ref_f64, absref, what):
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    bound = np.maximum(np.abs(ref_f64), 2.0 ** -126) * 2.0 ** -7 + PER_ELEM * absref
    err = np.abs(got - ref_f64)
    assert (err <= bound).all(), f"{what}: max err/bound {(err / bound).max():.3f}"


def _tile_view(h: dict, r0: int, c0: int) -> dict:
    """The 128 x 128 block of a host view at stored rows r0.., columns c0.."""
    bs = h["bs"]
    return dict(codes=h["codes"][r0:r0 + 128, c0:c0 + 128], scales=h["scales"][r0:r0 + 128, c0 // bs:(c0 + 128) // bs],
                senc=None, bs=bs, fmt=h["fmt"])


def test_swiglu_ffn_full_sampled_tiles():
    T, d, f = 16384, 4096, 14336
    t = config_tensors("c4_swiglu")
    X, W13, W2, DY2 = to_dev(t["x"]), to_dev(t["w13"]), to_dev(t["w2"]), to_dev(t["dy2"])
    xr, _ = F.fp4_quantize(X, "mx", 3, 0)
    w13r, _ = F.fp4_quantize(W13, "mx", 3, F.FP4_FLAG_WEIGHT_2D)
    _, w2c = F.fp4_quantize(W2, "mx", 3, F.FP4_FLAG_WEIGHT_2D)
    dyr, _ = F.fp4_quantize(DY2, "mx", 3, F.FP4_FLAG_SR_ROW, sr_seed=3)
    del X, W13, W2, DY2
    h_tap = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
    a1, a3, hr, hc = F.fp4_swiglu_fwd(xr, w13r, f, h_tap=h_tap)
    # the backward's saved activations: seeded host values (a 1024-row block repeated)
    a1_in = np.tile(normal_bf16((1024, f), 2.0, 34, 1), (T // 1024, 1))
    a3_in = np.tile(normal_bf16((1024, f), 2.0, 34, 2), (T // 1024, 1))
    dh_tap = torch.empty((T, f), dtype=torch.bfloat16, device="cuda")
    da_tap = torch.empty((T, 2 * f), dtype=torch.bfloat16, device="cuda")
    rr, cc = F.fp4_swiglu_bwd(dyr, w2c, f, to_dev(a1_in), to_dev(a3_in), sr_seed=3, sr_offset=1, dh_tap=dh_tap,
                              da13_tap=da_tap)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    qx = oracle.quantize(t["x"], "mx", "row")
    qw13 = oracle.quantize(t["w13"], "mx", "row", weight2d=True)
    qdy = oracle.quantize(t["dy2"], "mx", "row", sr=True, seed=3, offset=0)
    qw2 = oracle.quantize(t["w2"], "mx", "col", weight2d=True)
    same_view(xr, qx, "X row")
    same_view(w13r, qw13, "W13 row")
    same_view(dyr, qdy, "dY2 row")
    same_view(w2c, qw2, "W2 col")
    g_hr, g_hc, g_rr, g_cc = mhost(hr), mhost(hc), mhost(rr), mhost(cc)
    rng = np.random.default_rng(10)
    for _ in range(4):
        m0 = int(rng.integers(0, T // 128)) * 128
        n0 = int(rng.integers(0, f // 128)) * 128
        mm, nn = np.meshgrid(np.arange(m0, m0 + 128), np.arange(n0, n0 + 128), indexing="ij")
        ms, ns = mm.ravel(), nn.ravel()
        # forward: a1, a3, h and both views of h on this tile
        c1, ab1 = oracle.gemm_sampled(qx, qw13, ms, ns)
        c3, ab3 = oracle.gemm_sampled(qx, qw13, ms, ns + f)
        c1, c3, ab1, ab3 = (v.reshape(128, 128) for v in (c1, c3, ab1, ab3))
        o_a1, o_a3 = oracle.round_bf16(c1), oracle.round_bf16(c3)
        o_h = oracle.swiglu_h(o_a1, o_a3)
        g_a1 = bits(a1[m0:m0 + 128, n0:n0 + 128])
        g_a3 = bits(a3[m0:m0 + 128, n0:n0 + 128])
        g_h = bits(h_tap[m0:m0 + 128, n0:n0 + 128])
        _bf16_close(g_a1, c1, ab1, "a1")
        _bf16_close(g_a3, c3, ab3, "a3")
        same_in = (g_a1 == o_a1) & (g_a3 == o_a3)
        assert np.abs(ordered(g_h) - ordered(o_h))[same_in].max() <= 1
        same_h = g_h == o_h
        assert_view_masked(_tile_view(g_hr, m0, n0), oracle.quantize(o_h, "mx", "row"), g_h, same_h, "Q_r(h)")
        assert_view_masked(_tile_view(g_hc, n0, m0), oracle.quantize(o_h, "mx", "col"), oriented(g_h, "col"),
                           oriented(same_h, "col"), "Q_c(h)")
        # backward: dh, [da1 | da3] and both views of them on this tile
        c, ab = oracle.gemm_sampled(qdy, qw2, ms, ns)
        c, ab = c.reshape(128, 128), ab.reshape(128, 128)
        o_dh = oracle.round_bf16(c)
        g_dh = bits(dh_tap[m0:m0 + 128, n0:n0 + 128])
        _bf16_close(g_dh, c, ab, "dh")
        o1, o3 = oracle.swiglu_bwd(o_dh, np.ascontiguousarray(a1_in[m0:m0 + 128, n0:n0 + 128]),
                                   np.ascontiguousarray(a3_in[m0:m0 + 128, n0:n0 + 128]))
        for half, o in ((0, o1), (1, o3)):
            c0 = half * f + n0
            g_da = bits(da_tap[m0:m0 + 128, c0:c0 + 128])
            same_dh = g_dh == o_dh
            assert np.abs(ordered(g_da) - ordered(o))[same_dh].max() <= 1
            same = g_da == o
            want_r = oracle.quantize(o, "mx", "row", sr=True, seed=3, offset=1, sr_origin=(m0, c0), sr_cols=2 * f)
            assert_view_masked(_tile_view(g_rr, m0, c0), want_r, g_da, same, f"Q_r(da{1 + 2 * half})")
            assert_view_masked(_tile_view(g_cc, c0, m0), oracle.quantize(o, "mx", "col"), oriented(g_da, "col"),
                               oriented(same, "col"), f"Q_c(da{1 + 2 * half})")


# ------------------------------------------------- 32-block hybrid stack ----
def test_stack32_hybrid_full_step():
    sh = BlockShape()
    st = FP4LinearStack(32, 27, sh, seed=5)
    x_h = normal_bf16((sh.T, sh.d), 1.0, 5, 1)
    x, dy = to_dev(x_h), to_dev(normal_bf16((sh.T, sh.d), 1e-4, 5, 2))
    dx = st.step(x, dy, sr_seed=5)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    assert torch.isfinite(dx.float()).all()
    b0, top = st.blocks[0], st.blocks[-1]
    assert b0.route == "nv_local" and top.route == "mx" and st.blocks[27].route == "mx"
    # the first producer of the stack against the oracle (g = 1): the same
    # producer run again with a tap of y gives the stack's views, and those
    # match the oracle's wherever the kernel's y equals the oracle's
    tap = torch.empty((sh.T, sh.d), dtype=torch.bfloat16, device="cuda")
    _, rstd, yr, yc = F.fp4_residual_rmsnorm_fwd(x, None, st.g1, "nv_local", eps=st.eps, y_tap=tap)
    for a, b, what in ((yr, b0.s["y1"][0], "y1 row"), (yc, b0.s["y1"][1], "y1 col")):
        torch.cuda.synchronize()
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales), what
    ones = np.full(sh.d, 0x3F80, np.uint16)
    _, o_rstd, o_y = oracle.residual_rmsnorm(x_h, np.zeros_like(x_h), ones, st.eps)
    assert np.abs(rstd.cpu().numpy().view(np.int32) - o_rstd.view(np.int32)).max() <= 2
    y = bits(tap)
    assert np.abs(ordered(y) - ordered(o_y)).max() <= 1
    same = y == o_y
    assert_view_masked(mhost(yr), oracle.quantize(o_y, "nv_local", "row"), y, same, "block 0 Q_r(y1)")
    assert_view_masked(mhost(yc), oracle.quantize(o_y, "nv_local", "col"), oriented(y, "col"), oriented(same, "col"),
                       "block 0 Q_c(y1)")
    # weight gradients from the retained views: the gradient views are shared
    # per route, so the ones left at the end belong to the last block of each
    # route that the backward pass visited (block 0 and the first MXFP4 block)
    for blk in (b0, st.blocks[27]):
        gv, s = st.gviews[blk.route], blk.s
        for name, a, b in (("w2", gv["dF"][1], s["h"][1]), ("w13", gv["da13"][1], s["y2"][1]),
                           ("o", gv["dr2"][1], s["attn"][1]), ("qkv", gv["dqkv"][1], s["y1"][1])):
            assert torch.equal(F.fp4_linear_wgrad(a, b), blk.dw[name]), f"{blk.route} block dW{name}"


# ------------------------------------------- operand-wise hybrid, W1 shape ----
def test_operand_hybrid_w1_full():
    """MXFP4 Fprop and Wgrad (plain H16 on the pair), CTA-local NVFP4 Dgrad
    with row SR, at the W1 shape (Sec. 3.3), as the benchmark's hybrid leg
    runs it."""
    T, di, do = 8192, 4096, 14336
    t = config_tensors("c2_mx_w1")
    ones = [1] * 16
    X, W, DY = to_dev(t["x"]), to_dev(t["w"]), to_dev(t["dy"])
    h16 = F.FP4_FLAG_HADAMARD16_COL
    xr, xc = F.fp4_quantize(X, "mx", 3, h16, hadamard_signs=ones)
    wr, wc = F.fp4_quantize_hybrid(W, "mx", "nv_local", 3, F.FP4_FLAG_WEIGHT_2D)
    dr, dc = F.fp4_quantize_hybrid(DY, "nv_local", "mx", 3, F.FP4_FLAG_SR_ROW | h16, sr_seed=4, sr_offset=0,
                                   hadamard_signs=ones)
    Y = F.fp4_linear_fprop(xr, wr)
    DX = F.fp4_linear_dgrad(dr, wc)
    DW = F.fp4_linear_wgrad(dc, xc)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    del X, W, DY
    s1 = np.ones(16, np.int8)
    ov = dict(xr=oracle.quantize(t["x"], "mx", "row"),
              xc=oracle.quantize(t["x"], "mx", "col", hadamard16=True, signs=s1),
              wr=oracle.quantize(t["w"], "mx", "row", weight2d=True),
              wc=oracle.quantize(t["w"], "nv_local", "col", weight2d=True),
              dr=oracle.quantize(t["dy"], "nv_local", "row", sr=True, seed=4, offset=0),
              dc=oracle.quantize(t["dy"], "mx", "col", hadamard16=True, signs=s1))
    for k, v in dict(xr=xr, xc=xc, wr=wr, wc=wc, dr=dr, dc=dc).items():
        same_view(v, ov[k], f"hybrid W1 {k}")
    rng = np.random.default_rng(12)
    check_sampled(Y, ov["xr"], ov["wr"], "hybrid Fprop (MX)", rng)
    check_sampled(DX, ov["dr"], ov["wc"], "hybrid Dgrad (CTA-local)", rng)
    check_sampled(DW, ov["dc"], ov["xc"], "hybrid Wgrad (MX, H16 pair)", rng)


# ------------------------------------------------- QKV producer with RoPE ----
def test_qkv_rope_full():
    """The Llama-3-8B QKV boundary (T 8192, d 4096, 32 query and 8 key/value
    heads of 128, sequences of 4096): the fused forward on sampled 128-row
    blocks against the oracle's binary64 contraction turned in binary64, and
    the backward producer's gradient and CTA-local views bit for bit."""
    T, d, hq, hkv, S, route = 8192, 4096, 32, 8, 4096, "nv_local"
    N = (hq + 2 * hkv) * 128
    x = normal_bf16((T, d), 1.0, 95, 1)
    w = normal_bf16((N, d), 0.02, 95, 2)
    xr, _ = F.fp4_quantize(to_dev(x), route, F.FP4_VIEW_ROW)
    wr, _ = F.fp4_quantize(to_dev(w), route, F.FP4_VIEW_ROW, F.FP4_FLAG_WEIGHT_2D)
    c, s = oracle.rope_tables(S, 128)
    cd, sd = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    q, k, v = F.fp4_qkv_rope_fwd(xr, wr, cd, sd, S, hq, hkv)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    ox, ow = oracle.quantize(x, route, "row"), oracle.quantize(w, route, "row", weight2d=True)
    same_view(xr, ox, "X row")
    rng = np.random.default_rng(14)
    for _ in range(2):
        t0 = int(rng.integers(0, T // 128)) * 128
        mm, nn = np.meshgrid(np.arange(t0, t0 + 128), np.arange(N), indexing="ij")
        ref, absref = oracle.gemm_sampled(ox, ow, mm.ravel(), nn.ravel())
        ref, absref = ref.reshape(128, N), absref.reshape(128, N)
        pos = np.arange(t0, t0 + 128) % S
        cp, sp = c[pos].astype(np.float64), s[pos].astype(np.float64)
        for h in (0, hq - 1, hq, hq + hkv - 1):  # first and last query and key heads
            a, b = ref[:, h * 128:h * 128 + 64], ref[:, h * 128 + 64:(h + 1) * 128]
            aa, ab = absref[:, h * 128:h * 128 + 64], absref[:, h * 128 + 64:(h + 1) * 128]
            want = np.concatenate([a * cp - b * sp, b * cp + a * sp], axis=1)
            mag = np.concatenate([np.abs(a) * np.abs(cp) + np.abs(b) * np.abs(sp),
                                  np.abs(b) * np.abs(cp) + np.abs(a) * np.abs(sp)], axis=1)
            tol = np.concatenate([aa * np.abs(cp) + ab * np.abs(sp), ab * np.abs(cp) + aa * np.abs(sp)], axis=1)
            src = q[h] if h < hq else k[h - hq]
            got = oracle.bf16_to_f32(bits(src[t0:t0 + 128])).astype(np.float64)
            assert (np.abs(got - want) <= 2.0 ** -7 * mag + 2.0 ** -17 * tol + 1e-30).all(), f"head {h}"
    del q, k, v
    dq = normal_bf16((hq, T, 128), 1e-4, 96, 1)
    dk = normal_bf16((hkv, T, 128), 1e-4, 96, 2)
    dv = normal_bf16((hkv, T, 128), 1e-4, 96, 3)
    rr, cc = F.fp4_qkv_rope_bwd(to_dev(dq), to_dev(dk), to_dev(dv), cd, sd, S, route, 3, sr=True, sr_seed=6,
                                sr_offset=0)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    want = oracle.qkv_rope_bwd(dq, dk, dv, S, c, s)
    same_view(rr, oracle.quantize(want, route, "row", sr=True, seed=6, offset=0), "dQKV row")
    same_view(cc, oracle.quantize(want, route, "col"), "dQKV col")
