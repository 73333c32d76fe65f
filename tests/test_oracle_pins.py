"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: exact rationals derived
by hand from the definition, closed forms, invariants the operation must obey,
exact rational brute force on tiny integer inputs, and an independent float64
evaluation through library softmax / matmul.  Each pin is chosen so that a
plausible slip in the oracle (dropped scale, wrong sign, transposed operand,
wrong GQA head index, wrong causal alignment, mask polarity, NaN on dead rows)
fails at least one of them.

Semantics follow FlagOS-OP PR #10 "feat: add sdpa_math operator": (out, P) of
the SDPA math backend; causal and attn_mask are mutually exclusive; a bool mask
means -inf masking; a fully masked row gives P = O = 0; GQA needs Hq % Hkv == 0.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import oracle_fwd, OracleError
from sdpa_forward_materialised_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
LN2 = math.log(2.0)


def _t(x, dtype=torch.float64):
    return torch.tensor(x, dtype=dtype)


def _frac_array(nested):
    return np.vectorize(lambda s: float(Fraction(s)))(np.array(nested, dtype=object)).astype(np.float64)


# --------------------------------------------------------------------------- exact rationals

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_rationals(case):
    q, k, v = _t(case["q"]), _t(case["k"]), _t(case["v"])
    mask = None
    if case.get("mask") is not None:
        raw = case["mask"]
        if case["mask_kind"] == "bool":
            mask = torch.tensor(raw, dtype=torch.bool)
        else:
            mask = torch.tensor(np.array(raw, dtype=object).astype(np.float64))
    O, P, lse = oracle_fwd(q, k, v, mask, is_causal=case["is_causal"], scale=LN2)
    np.testing.assert_allclose(P, _frac_array(case["P"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(O, _frac_array(case["O"]), rtol=0, atol=1e-13)


def test_exact_rational_brute_force():
    """Every q in {-1,0,1}^2 against every 2-key K in {-1,0,1}^(2x2), V fixed
    integers, scale = ln 2: P and O are exact rationals (powers of two)."""
    vals = (-1, 0, 1)
    vrows = [[3, -1], [-2, 5]]
    qs = list(itertools.product(vals, repeat=2))
    ks = list(itertools.product(vals, repeat=4))
    q = _t([[[list(qq) for qq in qs]]])                    # [1,1,9,2]
    for kk in ks:
        k = _t([[[[kk[0], kk[1]], [kk[2], kk[3]]]]])
        v = _t([[vrows]])
        O, P, _ = oracle_fwd(q, k, v, scale=LN2)
        for i, qq in enumerate(qs):
            n = [qq[0] * kk[0] + qq[1] * kk[1], qq[0] * kk[2] + qq[1] * kk[3]]
            w = [Fraction(2) ** nj for nj in n]
            z = sum(w)
            p = [wj / z for wj in w]
            o = [p[0] * vrows[0][e] + p[1] * vrows[1][e] for e in range(2)]
            assert np.allclose(P[0, 0, i], [float(x) for x in p], rtol=0, atol=1e-15)
            assert np.allclose(O[0, 0, i], [float(x) for x in o], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("D,scale", [(4, None), (16, 0.37), (64, 2.5)])
def test_two_key_logistic(D, scale):
    """With two keys, P[:,0] = 1 / (1 + exp(-scale * q.(k0 - k1))) -- pins the
    scale, the sign and which operand is which."""
    g = torch.Generator().manual_seed(11 + D)
    q = torch.randn(2, 3, 7, D, generator=g, dtype=torch.float64)
    k = torch.randn(2, 3, 2, D, generator=g, dtype=torch.float64)
    v = torch.randn(2, 3, 2, 5, generator=g, dtype=torch.float64)
    sc = (1.0 / math.sqrt(D)) if scale is None else scale
    O, P, lse = oracle_fwd(q, k, v, scale=scale)
    qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
    diff = np.einsum("bhid,bhd->bhi", qn, kn[:, :, 0] - kn[:, :, 1])
    p0 = 1.0 / (1.0 + np.exp(-sc * diff))
    np.testing.assert_allclose(P[..., 0], p0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(P[..., 1], 1.0 - p0, rtol=0, atol=1e-14)
    o = p0[..., None] * vn[:, :, None, 0, :] + (1 - p0)[..., None] * vn[:, :, None, 1, :]
    np.testing.assert_allclose(O, o, rtol=0, atol=1e-13)
    # lse of two keys: log(exp(s0) + exp(s1))
    s0 = sc * np.einsum("bhid,bhd->bhi", qn, kn[:, :, 0])
    s1 = sc * np.einsum("bhid,bhd->bhi", qn, kn[:, :, 1])
    np.testing.assert_allclose(lse, np.logaddexp(s0, s1), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_uniform(causal):
    """Q = 0 gives a uniform P over the allowed keys and O = their mean of V."""
    g = torch.Generator().manual_seed(5)
    B, H, S, D = 2, 3, 9, 8
    q = torch.zeros(B, H, S, D, dtype=torch.float64)
    k = torch.randn(B, H, S, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, H, S, 6, generator=g, dtype=torch.float64)
    O, P, _ = oracle_fwd(q, k, v, is_causal=causal)
    vn = v.numpy()
    for i in range(S):
        n = (i + 1) if causal else S
        np.testing.assert_allclose(P[:, :, i, :n], 1.0 / n, rtol=0, atol=1e-15)
        assert np.all(P[:, :, i, n:] == 0.0)
        np.testing.assert_allclose(O[:, :, i], vn[:, :, :n].mean(axis=2), rtol=0, atol=1e-14)


def test_single_allowed_key_is_one_hot():
    """A bool mask keeping exactly one key per row: P is one-hot, O is that V row."""
    g = torch.Generator().manual_seed(6)
    B, H, Sq, Skv, D = 2, 2, 5, 11, 4
    q, k, v = (torch.randn(B, H, n, D, generator=g, dtype=torch.float64) for n in (Sq, Skv, Skv))
    pick = torch.randint(0, Skv, (B, H, Sq), generator=g)
    mask = torch.zeros(B, H, Sq, Skv, dtype=torch.bool)
    mask.scatter_(3, pick[..., None], True)
    O, P, _ = oracle_fwd(q, k, v, mask)
    np.testing.assert_array_equal(P, mask.double().numpy())
    exp_o = torch.gather(v, 2, pick[..., None].expand(B, H, Sq, D)).numpy()
    np.testing.assert_array_equal(O, exp_o)


def test_causal_row0_and_upper_triangle():
    g = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn(2, 4, 33, 16, generator=g, dtype=torch.float64) for _ in range(3))
    O, P, _ = oracle_fwd(q, k, v, is_causal=True)
    np.testing.assert_array_equal(O[:, :, 0], v.numpy()[:, :, 0])
    iu = np.triu_indices(33, k=1)
    assert np.all(P[:, :, iu[0], iu[1]] == 0.0)


def test_additive_log_weights_closed_form():
    """Q = 0 with an additive mask log(w): P = w / sum(w) (pins the additive path)."""
    g = torch.Generator().manual_seed(8)
    Skv = 13
    w = torch.rand(1, 1, 4, Skv, generator=g, dtype=torch.float64) + 0.1
    q = torch.zeros(1, 1, 4, 3, dtype=torch.float64)
    k = torch.randn(1, 1, Skv, 3, generator=g, dtype=torch.float64)
    v = torch.randn(1, 1, Skv, 2, generator=g, dtype=torch.float64)
    O, P, _ = oracle_fwd(q, k, v, torch.log(w))
    wn = w.numpy()
    np.testing.assert_allclose(P, wn / wn.sum(-1, keepdims=True), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- invariants

def _rand(seed, B, Hq, Hkv, Sq, Skv, D, Dv=None):
    g = torch.Generator().manual_seed(seed)
    Dv = D if Dv is None else Dv
    return (torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float64),
            torch.randn(B, Hkv, Skv, D, generator=g, dtype=torch.float64),
            torch.randn(B, Hkv, Skv, Dv, generator=g, dtype=torch.float64))


@pytest.mark.parametrize("shape", [(1, 2, 2, 17, 17, 8), (2, 4, 1, 5, 31, 16), (1, 3, 3, 40, 9, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_nonnegative(shape, causal):
    q, k, v = _rand(21, *shape)
    O, P, lse = oracle_fwd(q, k, v, is_causal=causal)
    Sq, Skv = shape[3], shape[4]
    rows = P.sum(-1)
    alive = np.ones_like(rows, dtype=bool)
    if causal and Skv == 0:
        alive[:] = False
    np.testing.assert_allclose(rows[alive], 1.0, rtol=0, atol=1e-12)
    assert np.all(P >= 0.0)
    assert np.all(np.isfinite(lse))


def test_fully_masked_rows_are_zero_bool_and_additive():
    q, k, v = _rand(22, 2, 2, 2, 6, 10, 8)
    mask = torch.ones(2, 1, 6, 10, dtype=torch.bool)
    mask[0, 0, 2] = False
    mask[1, 0, 5] = False
    O, P, lse = oracle_fwd(q, k, v, mask)
    for b, i in [(0, 2), (1, 5)]:
        assert np.all(P[b, :, i] == 0.0) and np.all(O[b, :, i] == 0.0)
        assert np.all(np.isneginf(lse[b, :, i]))
    add = torch.zeros(2, 1, 6, 10, dtype=torch.float64).masked_fill(~mask, float("-inf"))
    O2, P2, _ = oracle_fwd(q, k, v, add)
    np.testing.assert_array_equal(P2, P)
    np.testing.assert_array_equal(O2, O)
    assert not np.isnan(P).any() and not np.isnan(O).any()


def test_gqa_equals_repeated_kv_heads():
    """Query head h reads kv head h // (Hq/Hkv): same as repeat_interleave of K/V."""
    q, k, v = _rand(23, 2, 8, 2, 7, 12, 8, 5)
    O, P, _ = oracle_fwd(q, k, v)
    kr, vr = k.repeat_interleave(4, dim=1), v.repeat_interleave(4, dim=1)
    O2, P2, _ = oracle_fwd(q, kr, vr)
    np.testing.assert_array_equal(P, P2)
    np.testing.assert_array_equal(O, O2)
    # and differs from the modulo mapping (guards against h % Hkv)
    km = k.repeat(1, 4, 1, 1)
    _, P3, _ = oracle_fwd(q, km, v.repeat(1, 4, 1, 1))
    assert np.abs(P3 - P).max() > 1e-3


def test_all_true_mask_equals_no_mask_and_polarity():
    q, k, v = _rand(24, 1, 2, 2, 8, 8, 4)
    O, P, _ = oracle_fwd(q, k, v)
    O1, P1, _ = oracle_fwd(q, k, v, torch.ones(1, 1, 8, 8, dtype=torch.bool))
    np.testing.assert_array_equal(P, P1)
    np.testing.assert_array_equal(O, O1)
    # False masks (True keeps): masking key 0 everywhere zeroes column 0
    m = torch.ones(1, 1, 8, 8, dtype=torch.bool)
    m[..., 0] = False
    _, P2, _ = oracle_fwd(q, k, v, m)
    assert np.all(P2[..., 0] == 0.0) and np.all(P2[..., 1:] > 0.0)


@pytest.mark.parametrize("Sq,Skv", [(9, 9), (3, 7), (7, 3)])
def test_causal_equals_top_left_tril_mask(Sq, Skv):
    q, k, v = _rand(25, 1, 2, 2, Sq, Skv, 4)
    O, P, _ = oracle_fwd(q, k, v, is_causal=True)
    tril = torch.ones(Sq, Skv, dtype=torch.bool).tril()[None, None]
    O2, P2, _ = oracle_fwd(q, k, v, tril)
    np.testing.assert_array_equal(P, P2)
    np.testing.assert_array_equal(O, O2)


def test_mask_broadcast_equals_explicit_expansion():
    q, k, v = _rand(26, 2, 3, 3, 5, 6, 4)
    g = torch.Generator().manual_seed(3)
    m = torch.rand(1, 1, 5, 6, generator=g) < 0.7
    O, P, _ = oracle_fwd(q, k, v, m)
    O2, P2, _ = oracle_fwd(q, k, v, m.expand(2, 3, 5, 6).clone())
    np.testing.assert_array_equal(P, P2)
    np.testing.assert_array_equal(O, O2)
    mb = torch.rand(2, 1, 5, 6, generator=g) < 0.7
    O3, P3, _ = oracle_fwd(q, k, v, mb)
    O4, P4, _ = oracle_fwd(q, k, v, mb.expand(2, 3, 5, 6).clone())
    np.testing.assert_array_equal(P3, P4)
    np.testing.assert_array_equal(O3, O4)


def test_key_permutation_permutes_columns_only():
    q, k, v = _rand(27, 1, 2, 2, 6, 10, 4)
    perm = torch.randperm(10, generator=torch.Generator().manual_seed(1))
    O, P, _ = oracle_fwd(q, k, v)
    O2, P2, _ = oracle_fwd(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(P2, P[..., perm.numpy()], rtol=0, atol=1e-15)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-14)


def test_additive_row_shift_invariance_and_scale_equivalence():
    q, k, v = _rand(28, 1, 2, 2, 5, 7, 4)
    c = torch.arange(5, dtype=torch.float64).view(1, 1, 5, 1).expand(1, 1, 5, 7) * 3.0
    O, P, _ = oracle_fwd(q, k, v, torch.zeros(1, 1, 5, 7, dtype=torch.float64))
    O2, P2, _ = oracle_fwd(q, k, v, c.clone())
    np.testing.assert_allclose(P2, P, rtol=0, atol=1e-14)
    # scale * (q . k) == (scale/2) * ((2q) . k)
    O3, P3, _ = oracle_fwd(2 * q, k, v, scale=0.25)
    O4, P4, _ = oracle_fwd(q, k, v, scale=0.5)
    np.testing.assert_allclose(P3, P4, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- library cross-check

def _library_reference(q, k, v, mask, causal, scale):
    """Independent float64 evaluation with torch.softmax / torch.matmul."""
    q, k, v = q.double(), k.double(), v.double()
    g = q.shape[1] // k.shape[1]
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    s = torch.matmul(q, kr.transpose(-1, -2)) * scale
    if causal:
        Sq, Skv = s.shape[-2:]
        s = s.masked_fill(~torch.ones(Sq, Skv, dtype=torch.bool).tril(), float("-inf"))
    if mask is not None:
        if mask.dtype == torch.bool:
            s = s.masked_fill(~mask, float("-inf"))
        else:
            s = s + mask.double()
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)       # fully masked rows -> 0
    return torch.matmul(p, vr).numpy(), p.numpy()


def _small(w: W.Workload):
    # same recipe, shrunk so the CPU check stays fast
    S = min(w.Sq, 80)
    Skv = min(w.Skv, 96)
    if w.is_causal:
        Skv = S
    return W.make_custom(w.seed, min(w.B, 2), min(w.Hq, 4), min(w.Hkv, 4) if w.Hq != w.Hkv else min(w.Hq, 4),
                         S, Skv, w.D, w.dtype, mask=("bool" if w.mask else None))


@pytest.mark.parametrize("w", W.ALL, ids=lambda w: w.name)
def test_library_crosscheck(w):
    if w.name == "tiny_f32":
        q, k, v, m = W.make_inputs(w)
    else:
        q, k, v, m = _small(w)
    O, P, _ = oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale)
    O2, P2 = _library_reference(q, k, v, m, w.is_causal, w.scale)
    np.testing.assert_allclose(P, P2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)


def test_library_crosscheck_additive_mask():
    q, k, v, m = W.make_custom(31, 2, 4, 2, 19, 23, 16, "f32", mask="additive", mask_h=4)
    O, P, _ = oracle_fwd(q, k, v, m, scale=0.3)
    O2, P2 = _library_reference(q, k, v, m, False, 0.3)
    np.testing.assert_allclose(P, P2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- host logic

def test_errors_follow_the_fixed_semantics():
    q, k, v = _rand(29, 1, 3, 2, 4, 4, 4)
    with pytest.raises(OracleError):
        oracle_fwd(q, k, v)                              # 3 % 2 != 0
    q, k, v = _rand(29, 1, 2, 2, 4, 4, 4)
    with pytest.raises(OracleError):
        oracle_fwd(q, k, v, torch.ones(1, 1, 4, 4, dtype=torch.bool), is_causal=True)


def test_row_subset_and_thread_count():
    q, k, v = _rand(30, 2, 4, 2, 11, 13, 8)
    O, P, lse = oracle_fwd(q, k, v, is_causal=True)
    rows = np.array([0, 5, 17, 2 * 4 * 11 - 1, 40])
    Or, Pr, lr = oracle_fwd(q, k, v, is_causal=True, rows=rows, nthreads=3)
    np.testing.assert_array_equal(Or, O.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(Pr, P.reshape(-1, 13)[rows])
    np.testing.assert_array_equal(lr, lse.reshape(-1)[rows])
    O4, P4, _ = oracle_fwd(q, k, v, is_causal=True, nthreads=4)
    np.testing.assert_array_equal(O4, O)
    np.testing.assert_array_equal(P4, P)


def test_empty_sizes():
    q, k, v = _rand(31, 1, 2, 2, 0, 5, 4)
    O, P, lse = oracle_fwd(q, k, v)
    assert O.shape == (1, 2, 0, 4) and P.shape == (1, 2, 0, 5)
    q, k, v = _rand(31, 1, 2, 2, 3, 0, 4)
    O, P, lse = oracle_fwd(q, k, v)
    assert P.shape == (1, 2, 3, 0) and np.all(O == 0.0) and np.all(np.isneginf(lse))


def test_tail_workload_structure():
    """The tail workload's mask keeps ~80% of keys and has 5% dead query rows."""
    q, k, v, m = W.make_inputs(W.TAIL100)
    assert m.shape == (4, 1, 100, 100) and m.dtype == torch.bool
    dead = (~m.any(-1)).sum().item()
    assert dead == 20
    keep = m.float().mean().item()
    assert 0.74 < keep < 0.80
    O, P, _ = oracle_fwd(q, k, v, m)
    dead_rows = ~m.any(-1).expand(4, 8, 100).numpy()
    assert np.all(P[dead_rows] == 0.0) and np.all(O[dead_rows] == 0.0)
