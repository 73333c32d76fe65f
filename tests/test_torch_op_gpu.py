"""GPU checks of the PyTorch operator: forward parity with the fp64 oracle,
autograd through both outputs against the oracle backward, the aten override
under F.scaled_dot_product_attention (MATH backend), and torch.library's own
operator checks."""
import math

import numpy as np
import pytest
import torch

from sdpa_forward_materialised_gb300 import torch_op as T
from sdpa_forward_materialised_gb300 import workloads as W
from oracle import oracle_bwd, oracle_fwd
from parity_util import TOL, ulp

pytestmark = pytest.mark.gpu


def _close(got, ref, dtype, what, rel=0.0):
    g = got.detach().double().cpu().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, what
    if r.size == 0:
        return
    allow = TOL[dtype] + ulp(r, dtype) + rel * np.abs(r).max()
    bad = np.abs(g - r) > allow
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond tolerance, max err {np.abs(g - r).max():.3e}"


CASES = [
    # B, Hq, Hkv, Sq, Skv, D, dtype, causal, mask
    (1, 4, 4, 130, 130, 64, "f16", True, None),
    (2, 8, 2, 64, 200, 128, "bf16", False, None),
    (2, 2, 2, 100, 100, 64, "f16", False, "bool"),
    (1, 2, 2, 40, 77, 32, "f32", False, "additive"),
]


@pytest.mark.parametrize("idx", range(len(CASES)), ids=lambda i: "x".join(str(x) for x in CASES[i]))
def test_op_forward_and_autograd_match_oracle(idx):
    B, Hq, Hkv, Sq, Skv, D, dt, causal, mk = CASES[idx]
    q, k, v, m = W.make_custom(700 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mk)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    md = m.cuda() if m is not None else None
    O, P = torch.ops.sdpa_gb300.sdpa_math(qd, kd, vd, md, causal, None)
    Or, Pr, _ = oracle_fwd(q, k, v, m, is_causal=causal, scale=scale)
    _close(O, Or, q.dtype, "O")
    _close(P, Pr, q.dtype, "P")
    g = torch.Generator().manual_seed(900 + idx)
    G = torch.randn(O.shape, generator=g).to(q.dtype)
    H = torch.randn(P.shape, generator=g).to(q.dtype)
    ((O.float() * G.cuda().float()).sum() + (P.float() * H.cuda().float()).sum()).backward()
    rq, rk, rv = oracle_bwd(q, k, v, P.detach().cpu(), G, H, scale=scale)
    _close(qd.grad, rq, q.dtype, "dq", 1e-5)
    _close(kd.grad, rk, q.dtype, "dk", 1e-5)
    _close(vd.grad, rv, q.dtype, "dv", 1e-5)


def test_aten_override_under_the_math_backend():
    from torch.nn.attention import SDPBackend, sdpa_kernel
    q, k, v, _ = W.make_custom(750, 2, 8, 2, 96, 96, 64, "f16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O_op, P_op = torch.ops.sdpa_gb300.sdpa_math(qd, kd, vd, None, True, None)
    T.enable_aten_override()
    try:
        O_at, P_at = torch.ops.aten._scaled_dot_product_attention_math(qd, kd, vd, is_causal=True, enable_gqa=True)
        assert torch.equal(O_at, O_op) and torch.equal(P_at, P_op)
        with torch.inference_mode():  # the autograd keys are skipped: the CUDA-key entry serves the call
            O_im, P_im = torch.ops.aten._scaled_dot_product_attention_math(qd, kd, vd, is_causal=True, enable_gqa=True)
        assert torch.equal(O_im, O_op) and torch.equal(P_im, P_op)
        qg, kg, vg = (t.clone().requires_grad_(True) for t in (qd, kd, vd))
        with sdpa_kernel(SDPBackend.MATH):
            out = torch.nn.functional.scaled_dot_product_attention(qg, kg, vg, is_causal=True, enable_gqa=True)
        assert torch.equal(out, O_op)
        Gd = torch.randn(out.shape, generator=torch.Generator().manual_seed(3)).to(q.dtype).cuda()
        out.backward(Gd)
        rq, rk, rv = oracle_bwd(q, k, v, P_op.cpu(), Gd.cpu(), None, scale=1.0 / 8.0)
        _close(qg.grad, rq, q.dtype, "dq", 1e-5)
        _close(kg.grad, rk, q.dtype, "dk", 1e-5)
        _close(vg.grad, rv, q.dtype, "dv", 1e-5)
        with pytest.raises(NotImplementedError, match="dropout"):
            torch.ops.aten._scaled_dot_product_attention_math(qd, kd, vd, dropout_p=0.1, enable_gqa=True)
    finally:
        T.disable_aten_override()
    assert not torch._C._dispatch_has_kernel_for_dispatch_key("aten::_scaled_dot_product_attention_math",
                                                               "AutogradCUDA")
    Or, _, _ = oracle_fwd(q, k, v, None, is_causal=True, scale=1.0 / 8.0)
    _close(O_op, Or, q.dtype, "O")


def test_torch_library_opcheck():
    q, k, v, m = W.make_custom(760, 1, 4, 2, 40, 56, 64, "f16", mask="bool")
    args = (q.cuda().requires_grad_(True), k.cuda().requires_grad_(True), v.cuda().requires_grad_(True),
            m.cuda(), False, 0.125)
    torch.library.opcheck(torch.ops.sdpa_gb300.sdpa_math.default, args,
                          test_utils=("test_schema", "test_autograd_registration", "test_faketensor"))
