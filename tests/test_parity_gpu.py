"""GPU-vs-oracle parity of the (O, P) forward, through the C ABI.

Every case draws seeded inputs once, runs the CUDA path (outputs pre-filled
with NaN so an unwritten element cannot pass) and compares with the fp64 CPU
oracle element by element: in full at sizes the oracle finishes in seconds
(several tiles plus a ragged tail), and on sampled rows at the benchmark
shapes, together with properties that hold at any size (row sums, the zero
causal triangle, zero fully masked rows).

Semantics: FlagOS-OP PR #10 "feat: add sdpa_math operator" -- (out, P) of the
SDPA math backend; causal and mask mutually exclusive; bool mask = -inf
masking; fully masked row -> P = O = 0; GQA with Hq % Hkv == 0.
"""
import math
import os

import numpy as np
import pytest
import torch

import sdpa_forward_materialised_gb300 as sm
from sdpa_forward_materialised_gb300 import workloads as W
from oracle import oracle_fwd
from parity_util import compare, o_allowance, row_sum_bound, sample_rows

pytestmark = pytest.mark.gpu

NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sm.load_library()


def _run(q, k, v, mask, causal, scale, variant="auto", lse=False):
    dev = torch.device("cuda")
    # device tensors are used as they are (views with broadcast strides included)
    qd, kd, vd = (t if t.is_cuda else t.to(dev) for t in (q, k, v))
    md = (mask if mask.is_cuda else mask.to(dev)) if mask is not None else None
    if md is not None:
        while md.dim() < 4:
            md = md.unsqueeze(0)
    B, Hq, Sq, _ = q.shape
    Skv, Dv = k.shape[2], v.shape[3]
    O = torch.full((B, Hq, Sq, Dv), float("nan"), dtype=q.dtype, device=dev)
    P = torch.full((B, Hq, Sq, Skv), float("nan"), dtype=q.dtype, device=dev)
    L = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=dev) if lse else None
    kind = sm.MASK_NONE if md is None else (sm.MASK_BOOL if md.dtype == torch.bool else sm.MASK_ADDITIVE)
    sm.sdpa_math_fwd_ex(qd, kd, vd, md, kind, causal, scale, O, P, L, variant)
    torch.cuda.synchronize()
    sm.sdpa_math_device_status()
    return O, P, L


def _full_check(q, k, v, mask, causal, scale, variant="auto", check_lse=True):
    O, P, L = _run(q, k, v, mask, causal, scale, variant, lse=check_lse)
    Or, Pr, lr = oracle_fwd(q, k, v, mask, is_causal=causal, scale=scale, nthreads=NTHREADS)
    so = compare(O, Or, q.dtype, "O", extra=o_allowance(Pr, v, q.shape[1] // k.shape[1], q.dtype))
    sp = compare(P, Pr, q.dtype, "P")
    if check_lse:
        Lg = L.double().cpu().numpy()
        dead = np.isneginf(lr)
        assert np.all(np.isneginf(Lg[dead])), "LSE of fully masked rows must be -inf"
        np.testing.assert_allclose(Lg[~dead], lr[~dead], rtol=2e-6, atol=2e-5)
    return so, sp


def _variants_for(q, k, v, mask, causal):
    """Every kernel family that accepts this call (the SIMT one always does)."""
    out = []
    for name in ("simt", "twopass", "paired", "fused", "onesweep", "decode", "split", "tcdecode"):
        try:
            sm.sdpa_math_plan(q, k, v, mask, is_causal=causal, variant=name)
            out.append(name)
        except sm.SdpaError:
            pass
    return out


# --------------------------------------------------------------------------- workloads

@pytest.mark.parametrize("w", [W.TINY, W.TAIL100, W.DECODE, W.DECODE_32K], ids=lambda w: w.name)
def test_workload_full_compare(w):
    q, k, v, m = W.make_inputs(w)
    for variant in ["auto"] + _variants_for(q, k, v, m, w.is_causal):
        _full_check(q, k, v, m, w.is_causal, w.scale, variant)


@pytest.mark.parametrize("w", [W.PREFILL_1K_D64, W.PREFILL_2K_D128, W.PREFILL_2K_D128_BF16, W.GQA_1K_D128],
                         ids=lambda w: w.name)
def test_workload_sampled_rows_and_properties(w):
    """Full benchmark shape in the benchmark's launch configuration (auto)."""
    q, k, v, m = W.make_inputs(w)
    O, P, L = _run(q, k, v, m, w.is_causal, w.scale, "auto", lse=True)
    rows = sample_rows(w.B, w.Hq, w.Sq, n_random=192, seed=w.seed)
    Or, Pr, lr = oracle_fwd(q, k, v, m, is_causal=w.is_causal, scale=w.scale, rows=rows, nthreads=NTHREADS)
    compare(O.reshape(-1, w.D)[torch.from_numpy(rows).cuda()], Or, q.dtype, "O rows",
            extra=o_allowance(Pr, v, w.Hq // w.Hkv, q.dtype, rows=rows, Hq=w.Hq, Sq=w.Sq))
    compare(P.reshape(-1, w.Skv)[torch.from_numpy(rows).cuda()], Pr, q.dtype, "P rows")
    np.testing.assert_allclose(L.reshape(-1)[torch.from_numpy(rows).cuda()].double().cpu().numpy(), lr,
                               rtol=2e-6, atol=2e-5)
    # properties over every row
    assert not torch.isnan(P).any() and not torch.isnan(O).any()
    sums = P.double().sum(-1)
    assert (sums - 1).abs().max().item() <= row_sum_bound(q.dtype, w.Skv)
    assert (P >= 0).all()
    if w.is_causal:
        upper = torch.triu(torch.ones(w.Sq, w.Skv, dtype=torch.bool, device=P.device), diagonal=1)
        assert (P[..., upper] == 0).all()


# --------------------------------------------------------------------------- small multi-tile cases

SMALL = [
    # B, Hq, Hkv, Sq, Skv, D, dtype, causal, mask
    (1, 2, 2, 300, 300, 64, "f16", True, None),
    (2, 4, 2, 257, 390, 128, "f16", False, None),
    (1, 8, 2, 200, 136, 128, "bf16", False, None),
    (1, 2, 1, 384, 384, 128, "bf16", True, None),
    (2, 2, 2, 130, 270, 64, "f16", False, "bool"),
    (1, 4, 4, 96, 200, 64, "bf16", False, "additive"),
    (1, 2, 2, 77, 93, 32, "f32", True, None),
    (2, 3, 3, 50, 61, 96, "f32", False, "bool"),
    (1, 4, 1, 1, 700, 128, "f16", False, None),
    (3, 8, 2, 2, 1000, 64, "bf16", False, None),
    (1, 2, 2, 640, 640, 64, "f16", False, None),
    # shapes the TMA path takes (P row pitch a multiple of 16 bytes)
    (1, 2, 2, 328, 328, 64, "f16", True, None),
    (2, 4, 1, 200, 264, 128, "bf16", True, None),
    (1, 2, 2, 264, 136, 64, "f16", True, None),
    (1, 2, 2, 136, 136, 64, "f16", False, "bool"),
    (1, 3, 3, 520, 648, 128, "f16", False, None),
    (2, 2, 2, 129, 1032, 64, "bf16", True, None),
    # shapes the fused single-sweep kernel takes (Skv <= 256), incl. P rows of
    # 200 bytes (no TMA) and a single key
    (2, 4, 2, 130, 256, 128, "f16", True, None),
    (1, 2, 2, 100, 100, 64, "bf16", False, "bool"),
    (1, 2, 1, 7, 1, 64, "f16", False, None),
    (1, 3, 3, 250, 129, 128, "bf16", False, "additive"),
    # the same kernel on a grid large enough to keep 128-row query tiles (small
    # grids take 32-row query groups): 4 * 16 * 2 tiles
    (4, 16, 4, 200, 100, 64, "f16", False, "bool"),
    # causal calls whose row blocks keep at most two live key tiles however
    # long the key sequence (the fused kernel writes the masked tail of P as
    # zeros), incl. a P row of odd length
    (1, 4, 2, 200, 1000, 128, "f16", True, None),
    (2, 2, 2, 256, 300, 64, "bf16", True, None),
    (1, 2, 1, 130, 1001, 64, "f16", True, None),
    # few rows per KV head over long key sequences (split-KV): ragged chunks
    # and V sub-tiles, masks with fully masked rows, causal rows that see one
    # key, 16 rows at D = 256, and fewer keys than CTAs in the cluster
    (1, 4, 1, 1, 5000, 128, "f16", False, None),
    (2, 8, 2, 2, 3001, 64, "bf16", False, "bool"),
    (1, 2, 2, 8, 2500, 128, "f32", False, "additive"),
    (1, 16, 1, 1, 4100, 256, "f16", False, None),
    (1, 2, 1, 6, 2200, 64, "f16", True, None),
    (1, 4, 1, 1, 10, 64, "f16", False, None),
    # the tensor-core decode kernel (D = 128): one-tile and multi-tile chunks,
    # 16 rows, a bool mask with dead rows, causal rows, bf16, fewer keys than CTAs
    (2, 8, 2, 1, 1152, 128, "f16", False, None),
    (1, 16, 1, 1, 3000, 128, "bf16", False, None),
    (2, 4, 2, 2, 777, 128, "f16", False, "bool"),
    (1, 2, 1, 5, 600, 128, "f16", True, None),
    (1, 4, 2, 1, 9, 128, "bf16", False, "additive"),
]


@pytest.mark.parametrize("idx", range(len(SMALL)), ids=lambda i: "x".join(str(x) for x in SMALL[i]))
def test_small_cases_every_variant(idx):
    B, Hq, Hkv, Sq, Skv, D, dt, causal, mask = SMALL[idx]
    q, k, v, m = W.make_custom(100 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mask)
    scale = 1.0 / math.sqrt(D)
    variants = _variants_for(q, k, v, m, causal)
    assert "simt" in variants
    for variant in variants:
        _full_check(q, k, v, m, causal, scale, variant)


# The one-sweep kernel's clusters are persistent over query blocks.  With the
# grid capped to two clusters every cluster walks many blocks, causal blocks
# whose short rows leave some cluster ranks without a key tile (those ranks
# still take part in the statistics exchange and the O reduction), and blocks
# of every cluster size up to 4 CTAs.
ONESWEEP_PERSISTENT = [
    (1, 3, 3, 640, 640, 64, "f16", True, None),       # 2 CTAs per cluster
    (1, 2, 1, 1040, 1040, 128, "bf16", True, None),   # 3
    (2, 2, 2, 520, 648, 64, "f16", False, "bool"),    # 2, every rank busy
    (1, 4, 2, 1000, 1000, 128, "f16", True, None),    # 2, GQA
    (1, 2, 2, 1600, 1600, 64, "f16", True, None),     # 4
]


@pytest.mark.parametrize("idx", range(len(ONESWEEP_PERSISTENT)),
                         ids=lambda i: "x".join(str(x) for x in ONESWEEP_PERSISTENT[i]))
@pytest.mark.parametrize("clusters", [1, 2])
def test_onesweep_persistent_clusters(idx, clusters, monkeypatch):
    B, Hq, Hkv, Sq, Skv, D, dt, causal, mask = ONESWEEP_PERSISTENT[idx]
    monkeypatch.setenv("SDPA_MATH_ONESWEEP_CLUSTERS", str(clusters))
    q, k, v, m = W.make_custom(300 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mask)
    scale = 1.0 / math.sqrt(D)
    _full_check(q, k, v, m, causal, scale, "onesweep")


# The decode family has two kernels: 16-bit calls with head dims of 32, 64,
# 128 or 256 stream K and V through bulk copies; SDPA_MATH_DECODE_KERNEL=cluster
# forces the register-K kernel, which otherwise serves fp32 and other head
# dims.  Both run on every shape below.
DECODE_SHAPES = [
    # B, Hq, Hkv, Sq, Skv, D, Dv, dtype, causal, mask
    (2, 8, 2, 1, 1152, 128, 128, "f16", False, None),
    (1, 4, 2, 1, 300, 32, 32, "f16", False, None),
    (1, 8, 1, 1, 900, 256, 256, "bf16", False, None),
    (1, 4, 1, 1, 333, 64, 128, "f16", False, "bool"),       # dead rows, D != Dv
    (2, 4, 2, 2, 777, 128, 128, "bf16", False, "additive"),
    (1, 2, 1, 5, 600, 128, 128, "f16", True, None),         # 10 rows; causal rows see 1..5 keys
    (1, 16, 1, 1, 2048, 64, 64, "f16", False, None),        # 16 rows, 256-key chunks
    (1, 4, 2, 1, 9, 128, 128, "bf16", False, None),         # fewer keys than one piece
]


@pytest.mark.parametrize("kernel", ["stream", "cluster"])
@pytest.mark.parametrize("idx", range(len(DECODE_SHAPES)), ids=lambda i: "x".join(str(x) for x in DECODE_SHAPES[i]))
def test_decode_kernels(idx, kernel, monkeypatch):
    B, Hq, Hkv, Sq, Skv, D, Dv, dt, causal, mask = DECODE_SHAPES[idx]
    if kernel == "cluster":
        monkeypatch.setenv("SDPA_MATH_DECODE_KERNEL", "cluster")
    else:
        monkeypatch.delenv("SDPA_MATH_DECODE_KERNEL", raising=False)
    q, k, v, m = W.make_custom(400 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mask, Dv=Dv)
    _full_check(q, k, v, m, causal, 1.0 / math.sqrt(D), "decode")


def test_decode_rows_not_back_to_back():
    """K/V stored [B, S, H, D] (row stride H*D): the streaming decode kernel
    copies them row by row."""
    q, k, v, _ = W.make_custom(410, 2, 8, 2, 1, 1152, 128, "f16")
    kt = k.transpose(1, 2).contiguous().transpose(1, 2)
    vt = v.transpose(1, 2).contiguous().transpose(1, 2)
    assert kt.stride(2) == 2 * 128
    O, P, _ = _run(q, kt, vt, None, False, 1.0 / math.sqrt(128), "decode")
    Or, Pr, _ = oracle_fwd(q, k, v, None, scale=1.0 / math.sqrt(128), nthreads=NTHREADS)
    compare(O, Or, q.dtype, "O", extra=o_allowance(Pr, v, 4, q.dtype))
    compare(P, Pr, q.dtype, "P")


# --------------------------------------------------------------------------- seeded random shapes

def _random_cases(n, seed):
    """Shapes drawn from a fixed seed: dtypes, head dims (80 and D != Dv reach
    the CUDA-core and register-K kernels only), GQA groups, decode-like rows
    over long key sequences, ragged lengths, causal calls and both mask kinds."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        dt = str(rng.choice(["f16", "bf16", "f32"], p=[0.45, 0.45, 0.10]))
        D = int(rng.choice([32, 64, 80, 128]))
        Dv = D if rng.random() < 0.85 else int(rng.choice([32, 64, 128]))
        Hkv, group = int(rng.choice([1, 2, 3])), int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        if rng.random() < 0.35:
            Sq, Skv = int(rng.integers(1, 5)), int(rng.integers(1, 1500))
        else:
            Sq, Skv = int(rng.integers(1, 300)), int(rng.integers(1, 600))
        causal = bool(rng.random() < 0.3)
        mask = None if causal or rng.random() < 0.5 else str(rng.choice(["bool", "additive"]))
        cases.append((B, Hkv * group, Hkv, Sq, Skv, D, Dv, dt, causal, mask))
    return cases


RANDOM = _random_cases(64, 2024)


@pytest.mark.parametrize("idx", range(len(RANDOM)), ids=lambda i: "x".join(str(x) for x in RANDOM[i]))
def test_random_shapes_every_variant(idx):
    B, Hq, Hkv, Sq, Skv, D, Dv, dt, causal, mask = RANDOM[idx]
    q, k, v, m = W.make_custom(900 + idx, B, Hq, Hkv, Sq, Skv, D, dt, mask=mask, Dv=Dv)
    scale = 1.0 / math.sqrt(D)
    Or, Pr, lr = oracle_fwd(q, k, v, m, is_causal=causal, scale=scale, nthreads=NTHREADS)
    dead = np.isneginf(lr)
    for variant in ["auto"] + _variants_for(q, k, v, m, causal):
        O, P, L = _run(q, k, v, m, causal, scale, variant, lse=True)
        compare(O, Or, q.dtype, f"O {variant}", extra=o_allowance(Pr, v, Hq // Hkv, q.dtype))
        compare(P, Pr, q.dtype, f"P {variant}")
        Lg = L.double().cpu().numpy()
        assert np.all(np.isneginf(Lg[dead])), f"{variant}: LSE of fully masked rows must be -inf"
        np.testing.assert_allclose(Lg[~dead], lr[~dead], rtol=2e-6, atol=2e-5)


# --------------------------------------------------------------------------- edge cases

def test_empty_query_is_a_noop():
    q, k, v, _ = W.make_custom(1, 1, 2, 2, 0, 16, 64, "f16")
    O, P, _ = _run(q, k, v, None, False, 0.125)
    assert O.numel() == 0 and P.numel() == 0


def test_zero_keys_give_zero_output():
    q, k, v, _ = W.make_custom(2, 1, 2, 2, 5, 0, 64, "f16")
    O, P, L = _run(q, k, v, None, False, 0.125, lse=True)
    assert (O == 0).all() and P.numel() == 0 and torch.isneginf(L).all()


@pytest.mark.parametrize("D,Dv", [(1, 1), (8, 24), (80, 80), (256, 256), (40, 200)])
def test_head_dims(D, Dv):
    q, k, v, _ = W.make_custom(3, 1, 2, 2, 70, 90, D, "f16", Dv=Dv)
    _full_check(q, k, v, None, True, 1.0 / math.sqrt(D))


@pytest.mark.parametrize("Sq,Skv", [(150, 170), (136, 264)])
def test_transposed_bshd_layout(Sq, Skv):
    """[B,S,H,D] storage viewed as [B,H,S,D] (stride(-1) == 1, no copy)."""
    q, k, v, _ = W.make_custom(4, 2, 4, 2, Sq, Skv, 64, "f16")
    qt = q.transpose(1, 2).contiguous().transpose(1, 2)
    kt = k.transpose(1, 2).contiguous().transpose(1, 2)
    vt = v.transpose(1, 2).contiguous().transpose(1, 2)
    assert not qt.is_contiguous()
    O, P, _ = _run(qt, kt, vt, None, False, 0.125)
    Or, Pr, _ = oracle_fwd(q, k, v, None, scale=0.125, nthreads=NTHREADS)
    compare(O, Or, q.dtype, "O", extra=o_allowance(Pr, v, 2, q.dtype))
    compare(P, Pr, q.dtype, "P")


@pytest.mark.parametrize("mshape", [(1, 1), (2, 1), (1, 4), (2, 4)])
def test_mask_broadcast_forms(mshape):
    q, k, v, _ = W.make_custom(5, 2, 4, 2, 40, 72, 64, "f16")
    g = torch.Generator().manual_seed(9)
    m = torch.rand(mshape[0], mshape[1], 40, 72, generator=g) < 0.6
    m[0, 0, 3] = False  # a fully masked row
    _full_check(q, k, v, m, False, 0.125)


def test_additive_mask_f32_and_neg_inf_rows():
    q, k, v, _ = W.make_custom(6, 1, 2, 2, 33, 65, 64, "bf16")
    g = torch.Generator().manual_seed(10)
    m = torch.randn(1, 2, 33, 65, generator=g, dtype=torch.float32)
    m[0, 1, 7] = float("-inf")
    m[0, 0, 2, :10] = float("-inf")
    _full_check(q, k, v, m, False, 0.2)


def test_all_rows_masked():
    q, k, v, _ = W.make_custom(7, 1, 2, 2, 20, 30, 64, "f16")
    m = torch.zeros(1, 1, 20, 30, dtype=torch.bool)
    O, P, L = _run(q, k, v, m, False, 0.125, lse=True)
    assert (O == 0).all() and (P == 0).all() and torch.isneginf(L).all()


def test_sdpa_math_wrapper_matches_direct_call():
    q, k, v, _ = W.make_custom(8, 1, 4, 2, 100, 120, 64, "f16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O, P = sm.sdpa_math(qd, kd, vd, is_causal=True)
    O2, P2, _ = _run(q, k, v, None, True, 0.125)
    assert torch.equal(O, O2) and torch.equal(P, P2)


def test_forced_unsupported_variant_is_an_error():
    q, k, v, _ = W.make_custom(9, 1, 2, 2, 16, 16, 64, "f32")
    with pytest.raises(sm.SdpaError) as ei:
        _run(q, k, v, None, False, 0.125, variant="twopass")
    assert ei.value.status == sm.SDPA_ERR_UNSUPPORTED


# --------------------------------------------------------------------------- broadcast (stride-0) input views

def _broadcast_views(form, q, k, v):
    """Device views of q, k, v with one dimension broadcast (stride 0)."""
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if form == "kv_batch":      # every batch reads batch 0's keys and values
        kd, vd = kd[:1].expand_as(kd), vd[:1].expand_as(vd)
    elif form == "kv_heads":    # every key/value head reads head 0
        kd, vd = kd[:, :1].expand_as(kd), vd[:, :1].expand_as(vd)
    elif form == "q_heads":     # every query head reads head 0's queries
        qd = qd[:, :1].expand_as(qd)
    elif form == "q_rows":      # every query row is row 0
        qd = qd[:, :, :1].expand_as(qd)
    return qd, kd, vd


BCAST_SHAPES = [
    # B, Hq, Hkv, Sq, Skv, D, dtype, causal
    (2, 4, 2, 200, 264, 128, "f16", False),   # two-pass / paired (TMA), SIMT
    (2, 4, 2, 130, 200, 64, "bf16", True),    # fused (cp.async), two-pass, SIMT
    (2, 8, 2, 1, 1152, 128, "f16", False),    # decode, split-KV, tensor-core decode (TMA), SIMT
]


@pytest.mark.parametrize("form", ["kv_batch", "kv_heads", "q_heads", "q_rows"])
@pytest.mark.parametrize("shape", range(len(BCAST_SHAPES)), ids=lambda i: "x".join(map(str, BCAST_SHAPES[i])))
def test_broadcast_input_views(shape, form):
    """Inputs that are expand()ed views (stride 0 over batch, heads or rows)
    run on every family that accepts them, without a copy, and match the
    oracle on the materialised inputs.  Families that read 128-row TMA tiles
    refuse broadcast rows (the plan says so); the others serve every form."""
    B, Hq, Hkv, Sq, Skv, D, dt, causal = BCAST_SHAPES[shape]
    if form == "q_rows" and Sq == 1:
        pytest.skip("a single query row has nothing to broadcast")
    q, k, v, _ = W.make_custom(700 + shape, B, Hq, Hkv, Sq, Skv, D, dt)
    qd, kd, vd = _broadcast_views(form, q, k, v)
    assert 0 in (qd.stride() + kd.stride() + vd.stride())
    variants = _variants_for(qd, kd, vd, None, causal)
    assert "simt" in variants
    if form == "q_rows":
        assert not {"twopass", "paired"} & set(variants)
    qc, kc, vc = (t.contiguous().cpu() for t in (qd, kd, vd))
    Or, Pr, _ = oracle_fwd(qc, kc, vc, None, is_causal=causal, scale=1.0 / math.sqrt(D), nthreads=NTHREADS)
    for variant in ["auto"] + variants:
        O, P, _ = _run(qd, kd, vd, None, causal, 1.0 / math.sqrt(D), variant)
        compare(O, Or, q.dtype, f"O {form} {variant}", extra=o_allowance(Pr, vc, Hq // Hkv, q.dtype))
        compare(P, Pr, q.dtype, f"P {form} {variant}")
