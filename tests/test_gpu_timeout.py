"""The GEMM's bounded waits: a wait that cannot be satisfied runs out, the
kernel reports FP4_ERR_TIMEOUT through the status word and returns, and the
context stays usable (the next contraction is correct).

The wait is made to run out without any fault: the test hook makes the
epilogue skip its first accumulator release, so the MMA thread's wait for the
accumulator before each CTA pair's second tile is never satisfied.  The shape
gives every CTA pair at least two tiles (N = 256 x 160 columns of 256-wide
tiles for one 256-row M block, more tiles than there are pairs of SMs)."""
import numpy as np
import pytest
import torch

import oracle
import fp4_quantized_linears_gb300 as F
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu


def to_dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def test_gemm_wait_runs_out_reports_timeout_and_recovers():
    M, N, K = 256, 256 * 160, 256
    a = normal_bf16((M, K), 1.0, 71, 1)
    b = normal_bf16((N, K), 0.05, 71, 2)
    ar, _ = F.fp4_quantize(to_dev(a), "mx", F.FP4_VIEW_ROW)
    br, _ = F.fp4_quantize(to_dev(b), "mx", F.FP4_VIEW_ROW)
    torch.cuda.synchronize()
    F.fp4_status_reset()
    assert F.fp4_status() == F.FP4_OK
    F.fp4_set_wait_limit(20_000_000)  # about 10 ms at 2 GHz
    F.fp4_test_skip_accumulator_release(True)
    try:
        F.fp4_linear_fprop(ar, br)
        torch.cuda.synchronize()
        assert F.fp4_status() == F.FP4_ERR_TIMEOUT
    finally:
        F.fp4_test_skip_accumulator_release(False)
        F.fp4_set_wait_limit(0)
    F.fp4_status_reset()
    assert F.fp4_status() == F.FP4_OK
    # the context is intact: the same contraction again matches the oracle
    c = F.fp4_linear_fprop(ar, br)
    torch.cuda.synchronize()
    assert F.fp4_status() == F.FP4_OK
    ha, hb = oracle.quantize(a, "mx", "row"), oracle.quantize(b, "mx", "row")
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, M, 20000), rng.integers(0, N, 20000)
    ref, absref = oracle.gemm_sampled(ha, hb, ms, ns)
    got = c.cpu().numpy()[ms, ns].astype(np.float64)
    assert (np.abs(got - ref) <= 2.0 ** -18 * absref + 1e-30).all()
