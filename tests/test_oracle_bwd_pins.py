"""Pins of the oracle's backward (CPU only).

The backward follows FlagOS-OP PR #10 (overview, A1 item: gradients through
both outputs, dout and dprobs; "2026-10-07 update: P800 fused backward": the
exact softmax Jacobian of the materialised map, GQA gradients reduced back to
the KV heads).  It is pinned against things other than itself:

* central finite differences of the (separately pinned) oracle forward, for
  L = sum(O * G) + sum(P * H) with random G, H, on plain, causal, bool-masked
  (with a fully masked row), additive-masked and GQA shapes;
* an independent float64 evaluation by torch autograd through an explicit
  masked softmax and matmuls;
* invariants: a dead row gets no gradient, dprobs = None equals dprobs = 0,
  and GQA equals repeated K/V heads with their gradients summed per group.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle_bwd, oracle_fwd


def _inputs(seed, B, Hq, Hkv, Sq, Skv, D, Dv=None):
    g = torch.Generator().manual_seed(seed)
    Dv = D if Dv is None else Dv
    q = torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Skv, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Skv, Dv, generator=g, dtype=torch.float64)
    G = torch.randn(B, Hq, Sq, Dv, generator=g, dtype=torch.float64)
    H = torch.randn(B, Hq, Sq, Skv, generator=g, dtype=torch.float64)
    return q, k, v, G, H


def _loss(q, k, v, G, H, mask, causal, scale):
    O, P, _ = oracle_fwd(q, k, v, mask, is_causal=causal, scale=scale)
    return float((O * G.numpy()).sum() + (P * H.numpy()).sum())


def _numeric_grad(x, f, eps=1e-6):
    out = np.zeros(x.shape)
    flat = x.view(-1)
    for n in range(flat.numel()):
        old = flat[n].item()
        flat[n] = old + eps
        fp = f()
        flat[n] = old - eps
        fm = f()
        flat[n] = old
        out.reshape(-1)[n] = (fp - fm) / (2 * eps)
    return out


def _bool_mask_with_dead_row(seed, B, Sq, Skv):
    g = torch.Generator().manual_seed(seed)
    m = torch.rand(B, 1, Sq, Skv, generator=g) < 0.7
    m[:, :, 0, 0] = True
    m[:, :, Sq - 1, :] = False  # a fully masked row
    return m


CASES = [
    # name, B, Hq, Hkv, Sq, Skv, D, Dv, causal, mask
    ("plain", 1, 2, 2, 3, 4, 3, 2, False, None),
    ("causal_sq_lt_skv", 1, 1, 1, 3, 5, 2, 2, True, None),
    ("causal_sq_gt_skv", 1, 1, 1, 4, 3, 2, 3, True, None),
    ("bool_dead_row", 2, 2, 1, 3, 4, 2, 2, False, "bool"),
    ("additive", 1, 2, 2, 3, 3, 2, 2, False, "additive"),
    ("gqa", 1, 4, 2, 2, 3, 2, 2, False, None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_finite_differences(case):
    name, B, Hq, Hkv, Sq, Skv, D, Dv, causal, mk = case
    q, k, v, G, H = _inputs(11, B, Hq, Hkv, Sq, Skv, D, Dv)
    scale = 0.7
    mask = None
    if mk == "bool":
        mask = _bool_mask_with_dead_row(5, B, Sq, Skv)
    elif mk == "additive":
        mask = torch.randn(1, 1, Sq, Skv, generator=torch.Generator().manual_seed(3), dtype=torch.float64)
    _, P, _ = oracle_fwd(q, k, v, mask, is_causal=causal, scale=scale)
    dq, dk, dv = oracle_bwd(q, k, v, P, G, H, scale=scale)
    f = lambda: _loss(q, k, v, G, H, mask, causal, scale)
    for x, ana, nm in ((q, dq, "dq"), (k, dk, "dk"), (v, dv, "dv")):
        num = _numeric_grad(x, f)
        assert np.abs(num - ana).max() <= 1e-6 * max(1.0, np.abs(num).max()), (nm, num, ana)


def _torch_reference(q, k, v, G, H, mask, causal, scale):
    """Independent float64 evaluation: explicit masked softmax and matmuls,
    differentiated by torch autograd (GQA by repeating the KV heads)."""
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    g = q.shape[1] // k.shape[1]
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    s = scale * q @ kr.transpose(-1, -2)
    Sq, Skv = s.shape[-2:]
    if causal:
        keep = torch.ones(Sq, Skv, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf")) if mask.dtype == torch.bool else s + mask
    P = torch.softmax(s, dim=-1).nan_to_num(0.0)  # a fully masked row gives P = 0
    O = P @ vr
    L = (O * G).sum() + (P * H).sum()
    L.backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_float64_autograd(case):
    name, B, Hq, Hkv, Sq, Skv, D, Dv, causal, mk = case
    q, k, v, G, H = _inputs(21, B, Hq, Hkv, Sq, Skv, D, Dv)
    scale = 0.9
    mask = None
    if mk == "bool":
        mask = _bool_mask_with_dead_row(6, B, Sq, Skv)
    elif mk == "additive":
        mask = torch.randn(1, 1, Sq, Skv, generator=torch.Generator().manual_seed(4), dtype=torch.float64)
    _, P, _ = oracle_fwd(q, k, v, mask, is_causal=causal, scale=scale)
    got = oracle_bwd(q, k, v, P, G, H, scale=scale)
    ref = _torch_reference(q, k, v, G, H, mask, causal, scale)
    for a, r in zip(got, ref):
        np.testing.assert_allclose(a, r, rtol=1e-10, atol=1e-12)


def test_dead_row_gets_no_gradient_and_none_equals_zero_dprobs():
    q, k, v, G, H = _inputs(31, 1, 2, 2, 4, 5, 3)
    mask = torch.ones(1, 1, 4, 5, dtype=torch.bool)
    mask[..., 2, :] = False
    _, P, _ = oracle_fwd(q, k, v, mask, scale=0.5)
    dq, dk, dv = oracle_bwd(q, k, v, P, G, H, scale=0.5)
    assert np.all(dq[:, :, 2, :] == 0.0)
    # no dprobs is the same as dprobs = 0
    a = oracle_bwd(q, k, v, P, G, None, scale=0.5)
    b = oracle_bwd(q, k, v, P, G, torch.zeros_like(H), scale=0.5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_gqa_equals_repeated_heads_summed():
    q, k, v, G, H = _inputs(41, 2, 6, 2, 3, 4, 3, 2)
    _, P, _ = oracle_fwd(q, k, v, scale=0.6)
    dq, dk, dv = oracle_bwd(q, k, v, P, G, H, scale=0.6)
    kr, vr = k.repeat_interleave(3, dim=1), v.repeat_interleave(3, dim=1)
    dq2, dk2, dv2 = oracle_bwd(q, kr, vr, P, G, H, scale=0.6)
    np.testing.assert_allclose(dq, dq2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(2, 2, 3, 4, 3).sum(axis=2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(2, 2, 3, 4, 2).sum(axis=2), rtol=1e-12, atol=1e-13)
