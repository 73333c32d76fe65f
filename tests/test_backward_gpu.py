"""GPU parity of the backward (sdpa_math_bwd) against the fp64 oracle backward.

Both sides get the same probability map: the oracle forward's P rounded to the
dtype (an oracle output, cast on the CPU), so the comparison measures only the
GPU's fp32 accumulation and the rounding of dq, dk, dv to the dtype.

Tolerance, per element: the forward's absolute tolerance for the dtype
(1e-5 f32, 2e-3 f16, 8e-3 bf16) plus one ulp of the dtype at |ref| (output
rounding) plus 1e-5 * max|ref| over the tensor (fp32 accumulation over up to
Skv terms of mixed sign).
"""
import math

import numpy as np
import pytest
import torch

import sdpa_forward_materialised_gb300 as sm
from sdpa_forward_materialised_gb300 import workloads as W
from oracle import oracle_bwd, oracle_fwd
from parity_util import TOL, ulp

pytestmark = pytest.mark.gpu


def _check(got, ref, dtype, what):
    g = got.detach().double().cpu().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, what
    assert not np.isnan(g).any(), f"{what}: NaN"
    if r.size == 0:
        return
    allow = TOL[dtype] + ulp(r, dtype) + 1e-5 * np.abs(r).max()
    err = np.abs(g - r)
    bad = err > allow
    if bad.any():
        idx = np.unravel_index(np.argmax(err - allow), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond tolerance; worst at {idx}: "
                             f"got {g[idx]!r} ref {r[idx]!r} allow {allow[idx]:.3e}")


CASES = [
    # B, Hq, Hkv, Sq, Skv, D, Dv, dtype, causal, mask, with_dprobs
    (1, 2, 2, 64, 64, 64, 64, "f32", False, None, True),
    (2, 4, 2, 100, 77, 64, 64, "f16", True, None, True),
    (1, 8, 2, 130, 200, 128, 128, "bf16", False, None, True),
    (2, 2, 2, 96, 130, 64, 64, "f16", False, "bool", True),
    (1, 3, 3, 40, 300, 32, 48, "f32", False, "additive", False),
    (1, 4, 1, 1, 257, 128, 128, "f16", False, None, True),
    (1, 2, 2, 33, 1, 256, 256, "bf16", False, None, True),
    # shapes the tensor-core kernels take (D == Dv in {64, 128}, P rows on
    # 16-byte boundaries): ragged query and key tiles, GQA, masks with fully
    # masked rows, no dprobs, a single query row
    (1, 2, 2, 64, 64, 64, 64, "f16", False, None, True),
    (2, 4, 2, 200, 136, 64, 64, "f16", True, None, True),
    (2, 2, 2, 96, 136, 64, 64, "f16", False, "bool", True),
    (1, 4, 1, 1, 264, 128, 128, "f16", False, None, True),
    (1, 2, 2, 257, 384, 128, 128, "bf16", True, None, False),
    (1, 3, 3, 40, 296, 64, 64, "bf16", False, "additive", True),
    (1, 8, 2, 384, 256, 128, 128, "f16", False, None, True),
]


def _tc_eligible(dt, D, Dv, Sq, Skv):
    # contiguous P: every row (and every head's first row) on a 16-byte boundary
    return dt in ("f16", "bf16") and D == Dv and D in (64, 128) and Skv % 8 == 0


@pytest.mark.parametrize("variant", ["simt", "tc"])
@pytest.mark.parametrize("idx", range(len(CASES)), ids=lambda i: "x".join(str(x) for x in CASES[i]))
def test_backward_matches_oracle(idx, variant):
    B, Hq, Hkv, Sq, Skv, D, Dv, dt, causal, mk, with_dp = CASES[idx]
    if variant == "tc" and not _tc_eligible(dt, D, Dv, Sq, Skv):
        pytest.skip("outside the tensor-core backward's conditions (covered by the host refusal test)")
    q, k, v, m = W.make_custom(300 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mk, Dv=Dv)
    scale = 1.0 / math.sqrt(D)
    _, Po, _ = oracle_fwd(q, k, v, m, is_causal=causal, scale=scale)
    P = torch.from_numpy(Po).to(q.dtype)  # the shared, dtype-rounded probability map
    g = torch.Generator().manual_seed(500 + idx)
    dout = torch.randn(B, Hq, Sq, Dv, generator=g).to(q.dtype)
    dprobs = torch.randn(B, Hq, Sq, Skv, generator=g).to(q.dtype) if with_dp else None
    dq, dk, dv = sm.sdpa_math_backward(q.cuda(), k.cuda(), v.cuda(), P.cuda(), dout.cuda(),
                                       dprobs.cuda() if dprobs is not None else None, scale=scale,
                                       variant=variant)
    sm.sdpa_math_device_status()
    rq, rk, rv = oracle_bwd(q, k, v, P, dout, dprobs, scale=scale)
    _check(dq, rq, q.dtype, "dq")
    _check(dk, rk, q.dtype, "dk")
    _check(dv, rv, q.dtype, "dv")


def test_backward_through_the_gpu_forward():
    """End to end: the GPU forward's own P feeds the GPU backward; the result
    matches the oracle backward on that same (GPU-rounded) map, and dead rows
    of a bool mask get exactly zero dq."""
    q, k, v, m = W.make_inputs(W.TAIL100)
    qd, kd, vd, md = q.cuda(), k.cuda(), v.cuda(), m.cuda()
    O, P = sm.sdpa_math(qd, kd, vd, md, scale=W.TAIL100.scale)
    g = torch.Generator().manual_seed(7)
    dout = torch.randn(O.shape, generator=g).to(q.dtype)
    dprobs = torch.randn(P.shape, generator=g).to(q.dtype)
    dq, dk, dv = sm.sdpa_math_backward(qd, kd, vd, P, dout.cuda(), dprobs.cuda(), scale=W.TAIL100.scale)
    sm.sdpa_math_device_status()
    rq, rk, rv = oracle_bwd(q, k, v, P.cpu(), dout, dprobs, scale=W.TAIL100.scale)
    _check(dq, rq, q.dtype, "dq")
    _check(dk, rk, q.dtype, "dk")
    _check(dv, rv, q.dtype, "dv")
    dead = ~m.expand(q.shape[0], q.shape[1], -1, -1).any(-1)  # [B, Hq, Sq] rows with every key masked
    assert dead.any()
    assert (dq.cpu()[dead] == 0).all()


def test_tensor_core_backward_through_the_gpu_forward():
    """A causal prefill slice: the GPU forward's P feeds the tensor-core
    backward (AUTO picks it here); the rows kernel's rowsum equals the oracle's
    sum_j P dP; the causal upper triangle contributes nothing."""
    q, k, v, _ = W.make_custom(77, 1, 4, 2, 320, 320, 128, "f16")
    scale = 1.0 / math.sqrt(128)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O, P = sm.sdpa_math(qd, kd, vd, is_causal=True, scale=scale)
    g = torch.Generator().manual_seed(8)
    dout = torch.randn(O.shape, generator=g).to(q.dtype)
    dprobs = torch.randn(P.shape, generator=g).to(q.dtype)
    dq, dk, dv = (torch.empty_like(t) for t in (qd, kd, vd))
    rowsum = torch.full(q.shape[:3], float("nan"), device="cuda")
    sm.sdpa_math_bwd(qd, kd, vd, P, dout.cuda(), dprobs.cuda(), scale, dq, dk, dv, rowsum)
    sm.sdpa_math_device_status()
    Pc = P.cpu()
    rq, rk, rv = oracle_bwd(q, k, v, Pc, dout, dprobs, scale=scale)
    _check(dq, rq, q.dtype, "dq")
    _check(dk, rk, q.dtype, "dk")
    _check(dv, rv, q.dtype, "dv")
    # rowsum = sum_j P (dout . v_j + dprobs), in fp64 from the same rounded operands
    Pd, vd64 = Pc.double(), v.double().repeat_interleave(2, dim=1)
    dP = dout.double() @ vd64.transpose(-1, -2) + dprobs.double()
    r_ref = (Pd * dP).sum(-1).numpy()
    np.testing.assert_allclose(rowsum.cpu().double().numpy(), r_ref, rtol=1e-4, atol=1e-3)
