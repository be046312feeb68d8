"""The block stack's stochastic-rounding state (Format-Aware Fusion for Fast
FP4 Pretraining, Sec. 2.5 and Appendix A.1: seeds and counter offsets are
state that must not repeat): every SR producer of a step gets its own Philox
counter offset, and consecutive steps never reuse one.  Runs on the CPU: the
library's entry points are replaced by recorders (host logic only), and the
oracle shows that two steps' offsets draw different codes."""
import numpy as np
import pytest
import torch

import fp4_quantized_linears_gb300.stack as stack_mod
import oracle
from fp4_quantized_linears_gb300.stack import BlockShape, FP4LinearStack, sr_offset
from synthetic import normal_bf16

ENTRY_POINTS = ("fp4_linear_dgrad", "fp4_linear_dgrad_rmsnorm", "fp4_linear_fprop", "fp4_linear_wgrad",
                "fp4_quantize", "fp4_residual_rmsnorm_bwd_parts", "fp4_residual_rmsnorm_fwd", "fp4_swiglu_bwd",
                "fp4_swiglu_fwd")


def test_offsets_are_distinct_and_step_major():
    seen = set()
    for step in (0, 1, 2, (1 << 32) - 1):
        for block in (0, 1, 31, 32):
            for k in range(5):
                o = sr_offset(step, block, k)
                assert o >> 32 == step and 0 <= o < 1 << 64
                assert o not in seen
                seen.add(o)
    with pytest.raises(ValueError):
        sr_offset(1 << 32, 0, 0)
    with pytest.raises(ValueError):
        sr_offset(0, 0, 16)


def test_stack_steps_draw_fresh_offsets(monkeypatch):
    calls = []

    def recorder(name):
        def f(*args, **kwargs):
            calls.append((name, args, kwargs))
            return None, None
        return f

    for name in ENTRY_POINTS:
        monkeypatch.setattr(stack_mod, name, recorder(name))
    used = []
    real = stack_mod.sr_offset

    def record_offset(step, block, k):
        o = real(step, block, k)
        used.append(o)
        return o

    monkeypatch.setattr(stack_mod, "sr_offset", record_offset)
    sh = BlockShape(T=128, d=128, f=256, qkv=256)
    st = FP4LinearStack(3, 2, sh, seed=1, device="cpu")
    x = torch.zeros((sh.T, sh.d), dtype=torch.bfloat16)
    per_step = []
    for _ in range(2):
        used.clear()
        st.step(x, x, sr_seed=9)
        per_step.append(list(used))
    # one offset for the top gradient and four SR producers per block
    assert all(len(u) == 1 + 4 * 3 for u in per_step)
    assert len(set(per_step[0])) == len(per_step[0])
    assert not set(per_step[0]) & set(per_step[1])
    assert st.step_index == 2
    # every SR call the stack made passed one of the recorded offsets
    sr_calls = [c for c in calls if c[0] in ("fp4_quantize", "fp4_swiglu_bwd", "fp4_residual_rmsnorm_bwd_parts")]
    passed = set()
    for name, args, kwargs in sr_calls:
        if "sr_offset" in kwargs:
            passed.add(kwargs["sr_offset"])
        elif name == "fp4_swiglu_bwd" and len(args) > 6:  # the MXFP4 route quantizes in the epilogue
            passed.add(args[6])
        elif name == "fp4_residual_rmsnorm_bwd_parts":
            passed.add(args[10])
    assert set(per_step[0]) | set(per_step[1]) <= passed


def test_consecutive_steps_round_differently():
    """The same gradient quantized with the offsets of one producer in two
    consecutive steps gives different stochastically rounded codes."""
    g = normal_bf16((128, 256), 1e-3, 3, 1)
    a = oracle.quantize(g, "mx", "row", sr=True, seed=9, offset=sr_offset(0, 4, 1))
    b = oracle.quantize(g, "mx", "row", sr=True, seed=9, offset=sr_offset(1, 4, 1))
    assert np.array_equal(a["scales"], b["scales"])
    assert (a["codes"] != b["codes"]).mean() > 0.05
