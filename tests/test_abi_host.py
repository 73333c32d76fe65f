"""C-ABI host checks (no GPU): the library loads, exports every declared
symbol, and rejects bad arguments on the host before any launch.

Argument rules follow FlagOS-OP PR #10 "feat: add sdpa_math operator"
(semantics item: causal and mask mutually exclusive, GQA divisibility; the
"_d1()" micro-optimisation item: only the innermost stride must be 1).
Valid argument sets are only ever passed to ``sdpa_math_plan``, which never
touches the GPU.
"""
import ctypes
import glob
import os
import re

import pytest
import torch

import sdpa_forward_materialised_gb300 as sm
from sdpa_forward_materialised_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sm.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(sdpa_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "sdpa_math_fwd" in names and "sdpa_math_last_error" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_abi_version(lib):
    assert sm.sdpa_math_abi_version() == 1


def _qkv(B=2, Hq=4, Hkv=2, Sq=33, Skv=47, D=64, Dv=None, dtype=torch.float16):
    Dv = D if Dv is None else Dv
    return (torch.zeros(B, Hq, Sq, D, dtype=dtype), torch.zeros(B, Hkv, Skv, D, dtype=dtype),
            torch.zeros(B, Hkv, Skv, Dv, dtype=dtype))


def _expect(status_name, fn, match=None):
    with pytest.raises(sm.SdpaError) as ei:
        fn()
    assert sm.STATUS[ei.value.status] == status_name, str(ei.value)
    if match:
        assert re.search(match, str(ei.value)), str(ei.value)


def test_plan_accepts_valid_calls(lib):
    q, k, v = _qkv()
    r = sm.sdpa_math_plan(q, k, v)
    assert r["launches"] == 1
    assert r["live_score_tiles"] == 2 * 4 * 1 * 1


def test_error_causal_with_mask(lib):
    q, k, v = _qkv()
    m = torch.ones(1, 1, 33, 47, dtype=torch.bool)
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v, m, is_causal=True),
            "mutually exclusive")


def test_error_gqa_not_divisible(lib):
    q, k, v = _qkv(Hq=6, Hkv=4)
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v), "divisible")


def test_error_dtype_mismatch(lib):
    q, k, v = _qkv()
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k.float(), v), "dtype")


def test_error_unsupported_dtype_and_head_dim(lib):
    q, k, v = _qkv(dtype=torch.float64)
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q, k, v))
    q, k, v = _qkv(D=264)
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q, k, v), "256")


def test_error_shapes(lib):
    q, k, v = _qkv()
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k[:1], v), "batch")
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v[:, :, :40]), "key length")
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k[..., :32], v), "head dim")
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v, out_shape=(2, 4, 33, 63)),
            "out must be")
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v, probs_shape=(2, 4, 33, 46)),
            "probs must be")


def test_error_innermost_stride(lib):
    q, k, v = _qkv()
    qt = torch.zeros(2, 4, 64, 33, dtype=torch.float16).transpose(2, 3)  # stride(-1) = 33
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(qt, k, v), "innermost stride")
    # a transposed [B, S, H, D] layout keeps stride(-1) == 1 and is accepted
    qs = torch.zeros(2, 33, 4, 64, dtype=torch.float16).transpose(1, 2)
    assert sm.sdpa_math_plan(qs, k, v)["launches"] == 1


def test_error_mask_shape_and_dtype(lib):
    q, k, v = _qkv()
    for shape in [(3, 1, 33, 47), (1, 2, 33, 47), (1, 1, 32, 47), (1, 1, 33, 48)]:
        _expect("SDPA_ERR_INVALID_ARGUMENT",
                lambda: sm.sdpa_math_plan(q, k, v, torch.ones(shape, dtype=torch.bool)), "mask shape")
    for shape in [(1, 1, 33, 47), (2, 1, 33, 47), (1, 4, 33, 47), (2, 4, 33, 47)]:
        assert sm.sdpa_math_plan(q, k, v, torch.ones(shape, dtype=torch.bool))["launches"] == 1
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_plan(q, k, v, torch.ones(1, 1, 33, 47, dtype=torch.bfloat16)),
            "additive mask")
    assert sm.sdpa_math_plan(q, k, v, torch.zeros(1, 1, 33, 47, dtype=torch.float32))["launches"] == 1


def test_error_scale_not_finite(lib):
    q, k, v = _qkv()
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v, scale=float("nan")), "finite")
    _expect("SDPA_ERR_INVALID_ARGUMENT", lambda: sm.sdpa_math_plan(q, k, v, scale=float("inf")), "finite")


def test_error_null_and_misaligned_pointers(lib):
    q, k, v = _qkv()
    out = torch.empty(2, 4, 33, 64, dtype=torch.float16)
    probs = torch.empty(2, 4, 33, 47, dtype=torch.float16)
    dq, dk, dv, do, dp = (sm.describe(t) for t in (q, k, v, out, probs))
    plan = sm.SdpaPlan()
    dq.data = None
    st = lib.sdpa_math_plan(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), None, 0, 0,
                            ctypes.c_float(0.125), ctypes.byref(do), ctypes.byref(dp), 0,
                            ctypes.byref(plan))
    assert st == sm.SDPA_ERR_INVALID_ARGUMENT and b"NULL" in lib.sdpa_math_last_error()
    dq = sm.describe(q)
    dq.data = q.data_ptr() + 1
    st = lib.sdpa_math_plan(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), None, 0, 0,
                            ctypes.c_float(0.125), ctypes.byref(do), ctypes.byref(dp), 0,
                            ctypes.byref(plan))
    assert st == sm.SDPA_ERR_INVALID_ARGUMENT and b"aligned" in lib.sdpa_math_last_error()
    # the fwd entry point validates the same way before touching CUDA
    st = lib.sdpa_math_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), None, 0, 0,
                           ctypes.c_float(0.125), ctypes.byref(do), ctypes.byref(dp), None)
    assert st == sm.SDPA_ERR_INVALID_ARGUMENT
    # mask kind without a mask, and a mask with kind NONE
    dq = sm.describe(q)
    st = lib.sdpa_math_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), None, 1, 0,
                           ctypes.c_float(0.125), ctypes.byref(do), ctypes.byref(dp), None)
    assert st == sm.SDPA_ERR_INVALID_ARGUMENT and b"mask" in lib.sdpa_math_last_error()
    dm = sm.describe(torch.ones(1, 1, 33, 47, dtype=torch.bool))
    st = lib.sdpa_math_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(dm), 0, 0,
                           ctypes.c_float(0.125), ctypes.byref(do), ctypes.byref(dp), None)
    assert st == sm.SDPA_ERR_INVALID_ARGUMENT


def test_dropout_rejected_by_binding():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="dropout"):
        sm.sdpa_math(q, k, v, dropout_p=0.1)


def test_last_error_is_cleared_on_success(lib):
    q, k, v = _qkv(Hq=6, Hkv=4)
    with pytest.raises(sm.SdpaError):
        sm.sdpa_math_plan(q, k, v)
    assert sm.sdpa_math_last_error() != ""
    q, k, v = _qkv()
    sm.sdpa_math_plan(q, k, v)
    assert sm.sdpa_math_last_error() == ""


@pytest.mark.parametrize("Sq,Skv,causal,expect", [
    (1024, 1024, True, 36), (2048, 2048, True, 136), (1024, 1024, False, 64),
    (100, 100, False, 1), (1, 1152, False, 9), (512, 512, True, 10), (128, 2048, False, 16),
    (0, 5, False, 0), (130, 300, True, 3)])
def test_live_tile_count(lib, Sq, Skv, causal, expect):
    """Live 128x128 score tiles after top-left causal truncation, per (b, h)."""
    q, k, v = _qkv(B=1, Hq=1, Hkv=1, Sq=Sq, Skv=Skv, D=8)
    assert sm.sdpa_math_plan(q, k, v, is_causal=causal)["live_score_tiles"] == expect


def test_f32_always_plans_simt(lib):
    q, k, v = _qkv(dtype=torch.float32)
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "simt"


# AUTO's kernel family per benchmark workload (host-only planning): the fused
# single-sweep kernel for P rows TMA cannot describe, the cluster decode kernel for few rows
# per KV head, the tensor-core split-KV kernel when those rows meet a long key
# sequence at D = 128 (the CUDA-core split-KV kernel at other head dims),
# the one-tile two-pass kernel for the causal prefills (1k D64: 64 query-tile
# pairs; 2k D128: causal rows of 16 key tiles), the paired layout for the GQA
# prefill, and the CUDA-core kernel for fp32.
@pytest.mark.parametrize("name,expect", [
    ("tiny_f32", "simt"), ("prefill1k_d64_f16", "twopass"), ("prefill2k_d128_f16", "twopass"),
    ("prefill2k_d128_bf16", "twopass"), ("gqa1k_d128_f16", "paired"), ("decode_skv1152_f16", "decode"),
    ("tail100_mask_f16", "fused"), ("decode_skv32k_f16", "tcdecode")])
def test_auto_choice_per_workload(lib, name, expect):
    from sdpa_forward_materialised_gb300 import workloads as W
    w = W.BY_NAME[name]
    q = torch.empty(w.B, w.Hq, w.Sq, w.D, dtype=w.torch_dtype)
    k = torch.empty(w.B, w.Hkv, w.Skv, w.D, dtype=w.torch_dtype)
    v = torch.empty(w.B, w.Hkv, w.Skv, w.D, dtype=w.torch_dtype)
    m = None
    if w.mask is not None:
        m = torch.empty(w.B, 1, w.Sq, w.Skv, dtype=torch.bool)
    assert sm.sdpa_math_plan(q, k, v, m, is_causal=w.is_causal)["variant"] == expect


# The tensor-core layout AUTO takes, pinned to the GB300 sweep (96 shapes,
# f16, L2 flushed, CUDA events) it was calibrated on; each case names the
# measured times (us) of the layouts involved.
@pytest.mark.parametrize("B,H,S,D,causal,expect", [
    (1, 8, 1024, 64, True, "onesweep"),    # onesweep 16.1, twopass 20.5: 64 blocks x 2 CTAs fit one wave
    (1, 8, 1024, 128, True, "onesweep"),   # onesweep 18.1, twopass 22.1
    (1, 16, 1024, 64, True, "twopass"),    # twopass 20.1, onesweep 22.2 (256 CTAs), paired 24.3 (64 pairs)
    (1, 8, 2048, 128, True, "twopass"),    # twopass 36.5, paired 42.6, onesweep 48.8
    (1, 16, 512, 64, True, "twopass"),     # twopass 16.0, paired 22.1 (one CTA per cluster: no onesweep)
    (1, 32, 1024, 64, True, "paired"),     # paired 26.2, twopass 30.3 (128 pairs)
    (1, 32, 1024, 128, True, "paired"),    # paired 30.3, twopass 32.4
    (1, 16, 2048, 64, True, "paired"),     # paired 39.2, twopass 41.3
    (1, 16, 2048, 128, True, "twopass"),   # twopass 45.8, paired 47.1 (100-step bench)
    (1, 64, 512, 128, True, "paired"),     # paired 24.2, twopass 24.9
    (1, 64, 2048, 64, True, "twopass"),    # twopass 134.8, paired 136.8 (512 pairs)
    (1, 64, 512, 64, False, "paired"),     # paired 20.1, twopass 26.2
    (1, 8, 1024, 64, False, "twopass"),    # twopass 20.1, paired 28.3 (no causal mask: no onesweep)
])
def test_auto_tensor_core_layout_follows_the_sweep(lib, B, H, S, D, causal, expect):
    q, k, v = _qkv(B=B, Hq=H, Hkv=H, Sq=S, Skv=S, D=D)
    assert sm.sdpa_math_plan(q, k, v, is_causal=causal)["variant"] == expect


def test_fused_takes_at_most_two_live_key_tiles_per_row_block(lib):
    """The fused kernel can serve a call when every row block keeps at most two
    live 128-key tiles after causal truncation (counted tiles, not Skv).  AUTO
    prefers the two-pass kernels wherever TMA describes the P rows (they
    measured faster on GB300) and takes the fused kernel for the rest."""
    q, k, v = _qkv(B=1, Hq=2, Hkv=2, Sq=100, Skv=256, D=64)
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "twopass"
    assert sm.sdpa_math_plan(q, k, v, variant="fused")["variant"] == "fused"
    q, k, v = _qkv(B=1, Hq=2, Hkv=2, Sq=100, Skv=100, D=64)       # 200-byte P rows: no TMA
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "fused"
    q, k, v = _qkv(B=1, Hq=2, Hkv=2, Sq=100, Skv=264, D=64)
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q, k, v, variant="fused"), "two live")
    # causal: 256 query rows see at most keys 0..255 whatever Skv is
    q, k, v = _qkv(B=1, Hq=2, Hkv=2, Sq=256, Skv=5001, D=64)
    r = sm.sdpa_math_plan(q, k, v, is_causal=True)
    assert r["variant"] == "fused" and r["live_score_tiles"] == 2 * 3
    q, k, v = _qkv(B=1, Hq=2, Hkv=2, Sq=257, Skv=5001, D=64)
    assert sm.sdpa_math_plan(q, k, v, is_causal=True)["variant"] == "simt"
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q, k, v, is_causal=True, variant="fused"), "two live")


def test_split_kv_limits(lib):
    """Few rows and a long key sequence go to a split-KV kernel while the
    scores of a key chunk fit shared memory: the tensor-core one at D = Dv =
    128 (f16 / bf16), the CUDA-core one at other head dims; past that, to the
    two-pass tensor-core kernel.  K and V are views whose rows overlap (row
    stride 16 bytes): planning reads no data."""
    def kv(Skv, D):
        base = torch.zeros((Skv - 1) * 8 + D, dtype=torch.float16)
        t = base.as_strided((1, 1, Skv, D), (0, 0, 8, 1))
        return t, t
    q = torch.zeros(1, 4, 1, 128, dtype=torch.float16)
    k, v = kv(2048, 128)
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "decode"
    k, v = kv(5000, 128)
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "tcdecode"
    assert sm.sdpa_math_plan(q, k, v, variant="split")["variant"] == "split"
    k, v = kv(131072, 128)                 # 4 rows x 8192 keys of scores: 128 KiB beside the 64 KiB K/V ring
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "tcdecode"
    assert sm.sdpa_math_plan(q, k, v, variant="split")["variant"] == "split"
    k, v = kv(1 << 18, 128)                # 256 KiB of scores: neither split kernel has room
    assert sm.sdpa_math_plan(q, k, v)["variant"] == "twopass"
    q64 = torch.zeros(1, 4, 1, 64, dtype=torch.float16)
    k, v = kv(5000, 64)
    assert sm.sdpa_math_plan(q64, k, v)["variant"] == "split"
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q64, k, v, variant="tcdecode"), "head dims must be 128")
    q16 = torch.zeros(1, 16, 1, 256, dtype=torch.float16)
    k, v = kv(4100, 256)
    assert sm.sdpa_math_plan(q16, k, v)["variant"] == "split"
    k, v = kv(1 << 16, 256)                # 16 rows x 4096 keys of scores: 256 KiB
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q16, k, v, variant="split"), "1/16 key chunk")
    q16 = torch.zeros(1, 16, 1, 128, dtype=torch.float16)
    k, v = kv(1 << 18, 128)                # 16 rows x 16384 keys of scores: 1 MiB
    assert sm.sdpa_math_plan(q16, k, v)["variant"] == "twopass"
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q16, k, v, variant="tcdecode"), "key chunk")
    q17 = torch.zeros(1, 17, 1, 128, dtype=torch.float16)
    k, v = kv(5000, 128)
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q17, k, v, variant="split"), "16 query rows")
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q17, k, v, variant="tcdecode"), "16 query rows")


def _bwd_args(B=1, Hq=4, Hkv=2, Sq=9, Skv=11, D=16, Dv=8, dtype=torch.float16):
    q = torch.zeros(B, Hq, Sq, D, dtype=dtype)
    k = torch.zeros(B, Hkv, Skv, D, dtype=dtype)
    v = torch.zeros(B, Hkv, Skv, Dv, dtype=dtype)
    P = torch.zeros(B, Hq, Sq, Skv, dtype=dtype)
    go = torch.zeros(B, Hq, Sq, Dv, dtype=dtype)
    return q, k, v, P, go, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)


def test_backward_variant_refusals(lib):
    """sdpa_math_bwd_ex: the tensor-core family refuses what it cannot serve
    (with the reason) before launching; unknown families are argument errors."""
    q, k, v, P, go, dq, dk, dv = _bwd_args(Hq=4, Hkv=2, Sq=9, Skv=16, D=64, Dv=64)
    rs = torch.zeros(1, 4, 9)
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P, go, None, 0.25, dq, dk, dv, rs, stream=0, variant=7),
            "backward variant")
    q2, k2, v2, P2, go2, dq2, dk2, dv2 = _bwd_args(Hq=4, Hkv=2, Sq=9, Skv=16, D=64, Dv=32)
    _expect("SDPA_ERR_UNSUPPORTED",
            lambda: sm.sdpa_math_bwd(q2, k2, v2, P2, go2, None, 0.25, dq2, dk2, dv2, rs, stream=0, variant="tc"),
            "D == Dv")
    q3, k3, v3, P3, go3, dq3, dk3, dv3 = _bwd_args(Hq=4, Hkv=2, Sq=9, Skv=13, D=64, Dv=64)
    _expect("SDPA_ERR_UNSUPPORTED",
            lambda: sm.sdpa_math_bwd(q3, k3, v3, P3, go3, None, 0.25, dq3, dk3, dv3, rs, stream=0, variant="tc"),
            "16-byte")
    q4, k4, v4, P4, go4, dq4, dk4, dv4 = _bwd_args(Hq=4, Hkv=2, Sq=9, Skv=16, D=64, Dv=64, dtype=torch.float32)
    _expect("SDPA_ERR_UNSUPPORTED",
            lambda: sm.sdpa_math_bwd(q4, k4, v4, P4, go4, None, 0.25, dq4, dk4, dv4, rs, stream=0, variant="tc"),
            "f16 or bf16")


def test_backward_argument_errors(lib):
    """Host-side checks of sdpa_math_bwd (they return before any launch; the
    stream handle is never used on these paths)."""
    q, k, v, P, go, dq, dk, dv = _bwd_args()
    rs = torch.zeros(1, 4, 9)
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P[..., :10], go, None, 0.25, dq, dk, dv, rs, stream=0), "probs")
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P, go[..., :7], None, 0.25, dq, dk, dv, rs, stream=0), "dout")
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P, go, None, 0.25, dq, dk[:, :1], dv, rs, stream=0), "dq, dk, dv")
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P, go, None, 0.25, dq, dk, dv, None, stream=0), "rowsum")
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P.float(), go, None, 0.25, dq, dk, dv, rs, stream=0), "dtype")
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q, k, v, P, go, P[..., :3], 0.25, dq, dk, dv, rs, stream=0), "dprobs")
    q6, k6, v6, P6, go6, dq6, dk6, dv6 = _bwd_args(Hq=6, Hkv=4)
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_bwd(q6, k6, v6, P6, go6, None, 0.25, dq6, dk6, dv6, rs, stream=0), "divisible")


def test_empty_value_head_dim_with_aligned_rows_plans_without_crashing(lib):
    """A V with Dv = 0 but a 16-byte row stride (a slice v[..., :0] of a
    contiguous tensor) over a long key sequence: the split-KV planners must
    refuse it (they size work per pair of value columns) rather than divide
    by zero on the host."""
    q = torch.zeros(1, 8, 1, 128, dtype=torch.float16)
    k = torch.zeros(1, 8, 4096, 128, dtype=torch.float16)
    vbase = torch.zeros(1, 8, 4096, 8, dtype=torch.float16)
    v = vbase[..., :0]
    assert v.stride(2) == 8
    r = sm.sdpa_math_plan(q, k, v)
    assert r["variant"] == "simt"
    for forced in ("decode", "split", "tcdecode"):
        _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(q, k, v, variant=forced))


def test_noalloc_backward_rejects_more_rows_than_its_array(lib):
    """sdpa_math_bwd_noalloc refuses, on the host and before any CUDA call,
    a call with more query rows (B*Hq*Sq) than its fixed row-sum array holds."""
    rows = sm.SDPA_BWD_NOALLOC_MAX_ROWS + 1
    q = torch.zeros(1, 1, rows, 1, dtype=torch.float16)
    k = torch.zeros(1, 1, 4, 1, dtype=torch.float16)
    P = torch.zeros(1, 1, rows, 4, dtype=torch.float16)
    _expect("SDPA_ERR_UNSUPPORTED",
            lambda: sm.sdpa_math_bwd_noalloc(q, k, k, P, q, None, 1.0, torch.empty_like(q), torch.empty_like(k),
                                             torch.empty_like(k), stream=0), "at most")


def test_outputs_must_not_overlap_themselves(lib):
    """An out or probs view with stride 0 over more than one element would be
    written by several threads at once: refused on the host."""
    q, k, v = _qkv()
    O = torch.zeros(2, 4, 1, 64, dtype=torch.float16).expand(2, 4, 33, 64)
    P = torch.zeros(2, 4, 33, 47, dtype=torch.float16)
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_plan(q, k, v, out=O, probs=P), "must not overlap")
    O = torch.zeros(2, 4, 33, 64, dtype=torch.float16)
    P = torch.zeros(1, 4, 33, 47, dtype=torch.float16).expand(2, 4, 33, 47)
    _expect("SDPA_ERR_INVALID_ARGUMENT",
            lambda: sm.sdpa_math_plan(q, k, v, out=O, probs=P), "must not overlap")


def test_broadcast_rows_refused_by_tma_families(lib):
    """Batch and head broadcasts are served by every family; broadcast rows
    (row stride 0) are refused by the families that read 128-row TMA tiles."""
    q, k, v = _qkv(B=2, Hq=4, Hkv=2, Sq=320, Skv=320, D=64)
    kb = k[:1].expand_as(k)
    assert sm.sdpa_math_plan(q, kb, v, variant="twopass")["variant"] == "twopass"
    qr = q[:, :, :1].expand_as(q)
    _expect("SDPA_ERR_UNSUPPORTED", lambda: sm.sdpa_math_plan(qr, k, v, variant="twopass"), "broadcast")
    assert sm.sdpa_math_plan(qr, k, v)["variant"] == "simt"
