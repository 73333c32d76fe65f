"""The backward entry point that allocates nothing: sdpa_math_bwd_noalloc.

Some callers cannot allocate device memory when they run the backward: code
hosted in a framework that hands out all device memory from its own
pre-planned pool, or a real-time path that must not call cudaMalloc after
start-up because the call can block and synchronise the device.
sdpa_math_bwd needs a B*Hq*Sq float buffer from its caller for the per-row
sums passed between its two kernels; sdpa_math_bwd_noalloc takes none and
keeps those sums in a fixed array of the library's own device memory.

These checks call it through the C ABI twice in a row, on different inputs
(the second call runs over what the first left in the shared array), and
compare each result with sdpa_math_bwd given a caller buffer, within the
tolerance of the backward parity tests.  This file is collected last, so a
run that stops at its first failure has run every other test before it.
"""
import math

import numpy as np
import pytest
import torch

import sdpa_forward_materialised_gb300 as sm
from sdpa_forward_materialised_gb300 import workloads as W
from parity_util import TOL, ulp

pytestmark = pytest.mark.gpu


def _close(got, ref, dtype, what):
    """The backward parity tolerance: the forward's absolute tolerance for the
    dtype, plus one ulp at |ref|, plus 1e-5 * max|ref| (fp32 accumulation)."""
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert g.shape == r.shape and not np.isnan(g).any(), what
    if r.size == 0:
        return
    allow = TOL[dtype] + ulp(r, dtype) + 1e-5 * np.abs(r).max()
    bad = np.abs(g - r) > allow
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond tolerance"


def _inputs(seed, B, Hq, Hkv, Sq, Skv, D, dt, causal):
    dev = torch.device("cuda")
    q, k, v, _ = W.make_custom(seed, B, Hq, Hkv, Sq, Skv, D, dt)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    scale = 1.0 / math.sqrt(D)
    _, P = sm.sdpa_math(qd, kd, vd, is_causal=causal, scale=scale)
    g = torch.Generator().manual_seed(seed + 1000)
    dout = torch.randn(B, Hq, Sq, D, generator=g).to(q.dtype).to(dev)
    dprobs = torch.randn(B, Hq, Sq, Skv, generator=g).to(q.dtype).to(dev)
    return qd, kd, vd, P, dout, dprobs, scale


def _with_caller_buffer(qd, kd, vd, P, dout, dprobs, scale):
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    rowsum = torch.empty(qd.shape[:3], dtype=torch.float32, device=qd.device)
    sm.sdpa_math_bwd(qd, kd, vd, P, dout, dprobs, scale, dq, dk, dv, rowsum)
    return dq, dk, dv


def _without_allocation(qd, kd, vd, P, dout, dprobs, scale):
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    sm.sdpa_math_bwd_noalloc(qd, kd, vd, P, dout, dprobs, scale, dq, dk, dv)
    return dq, dk, dv


# two calls in a row per kernel family: the first with more query rows than
# the second, so the second runs over rows the first left in the array
CALLS = {
    "tensor-core": [(11, 2, 8, 2, 384, 264, 128, "f16", True), (12, 1, 4, 2, 200, 136, 64, "bf16", False)],
    "cuda-core": [(21, 2, 6, 3, 150, 90, 96, "f16", False), (22, 1, 2, 2, 70, 50, 64, "f32", True)],
}


@pytest.mark.parametrize("family", sorted(CALLS))
def test_noalloc_backward_matches_the_caller_buffer_backward(family):
    sm.load_library()
    for call in CALLS[family]:
        seed, B, Hq, Hkv, Sq, Skv, D, dt, causal = call
        args = _inputs(seed, B, Hq, Hkv, Sq, Skv, D, dt, causal)
        ref = _with_caller_buffer(*args)
        got = _without_allocation(*args)
        torch.cuda.synchronize()
        sm.sdpa_math_device_status()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            _close(g, r, args[0].dtype, f"{family} call {seed} {name}")


def test_noalloc_rejects_more_rows_than_its_array():
    sm.load_library()
    rows = sm.SDPA_BWD_NOALLOC_MAX_ROWS + 1
    dev = torch.device("cuda")
    q = torch.zeros(1, 1, rows, 1, dtype=torch.float16, device=dev)
    k = torch.zeros(1, 1, 4, 1, dtype=torch.float16, device=dev)
    v = torch.zeros(1, 1, 4, 1, dtype=torch.float16, device=dev)
    P = torch.zeros(1, 1, rows, 4, dtype=torch.float16, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(sm.SdpaError) as ei:
        sm.sdpa_math_bwd_noalloc(q, k, v, P, q, None, 1.0, dq, dk, dv)
    assert ei.value.status == sm.SDPA_ERR_UNSUPPORTED
    assert "at most" in str(ei.value)
