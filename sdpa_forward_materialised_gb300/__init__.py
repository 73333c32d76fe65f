"""GB300 (sm_103a) materialised-probability SDPA forward: returns (O, P).

Thin ctypes binding over ``libsdpa_math.so`` (C ABI in ``include/sdpa_math.h``).
Everything here is argument marshalling: every step of the computation runs in
the library's CUDA kernels, and a missing library is an error, never a
fallback.  PyTorch provides device memory and the current stream only.

The operation is the SDPA math backend that returns both the output and the
attention-probability map (FlagOS-OP PR #10 "feat: add sdpa_math operator"):
P = softmax(scale * Q K^T + mask), O = P V, with causal and attn_mask mutually
exclusive, bool masks meaning -inf masking, fully masked rows giving P = O = 0,
GQA requiring Hq % Hkv == 0 and no dropout.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

from . import _build

__all__ = [
    "sdpa_math", "sdpa_math_fwd", "sdpa_math_fwd_ex", "sdpa_math_plan",
    "sdpa_math_bwd", "sdpa_math_backward", "BWD_VARIANTS", "sdpa_math_device_status", "sdpa_math_selftest_wait", "sdpa_math_last_error", "sdpa_math_abi_version",
    "SdpaError", "SdpaValueError", "load_library", "library_path", "VARIANTS", "STATUS",
]

SDPA_OK, SDPA_ERR_INVALID_ARGUMENT, SDPA_ERR_UNSUPPORTED, SDPA_ERR_CUDA, SDPA_ERR_TIMEOUT = range(5)
STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARGUMENT", 2: "SDPA_ERR_UNSUPPORTED",
          3: "SDPA_ERR_CUDA", 4: "SDPA_ERR_TIMEOUT"}
SDPA_F32, SDPA_F16, SDPA_BF16, SDPA_BOOL = range(4)
# Query rows (B*Hq*Sq) sdpa_math_bwd_noalloc serves (its fixed device row-sum array).
SDPA_BWD_NOALLOC_MAX_ROWS = 1 << 20
MASK_NONE, MASK_BOOL, MASK_ADDITIVE = range(3)
VARIANTS = {"auto": 0, "simt": 1, "twopass": 2, "fused": 3, "decode": 4, "paired": 5, "split": 6, "tcdecode": 7,
            "onesweep": 8}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}


class SdpaError(RuntimeError):
    """Non-OK status from the library; ``status`` holds the sdpa_status code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class SdpaValueError(SdpaError, ValueError):
    """Invalid or unsupported arguments (SDPA_ERR_INVALID_ARGUMENT / SDPA_ERR_UNSUPPORTED)."""


class SdpaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class SdpaPlan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("live_score_tiles", ctypes.c_int64),
                ("launches", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load ``libsdpa_math.so``.  Raises if it is not built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"the CUDA library {path} is not built; run "
                    "sdpa_forward_materialised_gb300._build.build() (nvcc, sm_103a)")
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        T = P(SdpaTensor)
        lib.sdpa_math_fwd.restype = ctypes.c_int
        lib.sdpa_math_fwd.argtypes = [T, T, T, T, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                      T, T, ctypes.c_void_p]
        lib.sdpa_math_fwd_ex.restype = ctypes.c_int
        lib.sdpa_math_fwd_ex.argtypes = [T, T, T, T, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                         T, T, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        lib.sdpa_math_plan.restype = ctypes.c_int
        lib.sdpa_math_plan.argtypes = [T, T, T, T, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                       T, T, ctypes.c_int, P(SdpaPlan)]
        lib.sdpa_math_device_status.restype = ctypes.c_int
        lib.sdpa_math_device_status.argtypes = [ctypes.c_void_p]
        lib.sdpa_math_bwd.restype = ctypes.c_int
        lib.sdpa_math_bwd.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_void_p,
                                      ctypes.c_void_p]
        lib.sdpa_math_bwd_ex.restype = ctypes.c_int
        lib.sdpa_math_bwd_ex.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_void_p,
                                         ctypes.c_int, ctypes.c_void_p]
        lib.sdpa_math_bwd_noalloc.restype = ctypes.c_int
        lib.sdpa_math_bwd_noalloc.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_void_p]
        lib.sdpa_math_selftest_wait.restype = ctypes.c_int
        lib.sdpa_math_selftest_wait.argtypes = [ctypes.c_void_p]
        lib.sdpa_math_last_error.restype = ctypes.c_char_p
        lib.sdpa_math_last_error.argtypes = []
        lib.sdpa_math_abi_version.restype = ctypes.c_int
        lib.sdpa_math_abi_version.argtypes = []
        _lib = lib
        return lib


def _dtype_code(dt) -> int:
    import torch
    m = {torch.float32: SDPA_F32, torch.float16: SDPA_F16, torch.bfloat16: SDPA_BF16,
         torch.bool: SDPA_BOOL}
    if dt not in m:
        return 99  # rejected by the library with SDPA_ERR_UNSUPPORTED
    return m[dt]


def describe(t, rank4: bool = True) -> SdpaTensor:
    """sdpa_tensor for a torch tensor (data pointer, dtype, extents, element strides)."""
    d = SdpaTensor()
    if t is None:
        return d
    shape, stride = list(t.shape), list(t.stride())
    while rank4 and len(shape) < 4:
        shape.insert(0, 1)
        stride.insert(0, 0)
    if len(shape) != 4:
        raise ValueError(f"expected a rank-4 tensor, got shape {tuple(t.shape)}")
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _dtype_code(t.dtype)
    for i in range(4):
        d.shape[i] = shape[i]
        d.stride[i] = stride[i]
    return d


def _raise(lib, status: int):
    msg = lib.sdpa_math_last_error().decode(errors="replace")
    if status in (SDPA_ERR_INVALID_ARGUMENT, SDPA_ERR_UNSUPPORTED):
        raise SdpaValueError(status, msg)
    raise SdpaError(status, msg)


def _mask_kind(mask) -> int:
    if mask is None:
        return MASK_NONE
    import torch
    return MASK_BOOL if mask.dtype == torch.bool else MASK_ADDITIVE


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return getattr(stream, "cuda_stream", stream)


def sdpa_math_fwd(q, k, v, mask, mask_kind, is_causal, scale, out, probs, stream=None):
    """Direct C-ABI call on caller-allocated device tensors (raises on error)."""
    lib = load_library()
    dq, dk, dv, do, dp = describe(q), describe(k), describe(v), describe(out), describe(probs)
    dm = describe(mask) if mask is not None else None
    st = lib.sdpa_math_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                           ctypes.byref(dm) if dm is not None else None, int(mask_kind),
                           int(bool(is_causal)), float(scale), ctypes.byref(do), ctypes.byref(dp),
                           _stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


def sdpa_math_fwd_ex(q, k, v, mask, mask_kind, is_causal, scale, out, probs, lse=None,
                     variant="auto", stream=None):
    """C-ABI call with a forced kernel family and an optional fp32 LSE output."""
    lib = load_library()
    dq, dk, dv, do, dp = describe(q), describe(k), describe(v), describe(out), describe(probs)
    dm = describe(mask) if mask is not None else None
    var = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    st = lib.sdpa_math_fwd_ex(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                              ctypes.byref(dm) if dm is not None else None, int(mask_kind),
                              int(bool(is_causal)), float(scale), ctypes.byref(do), ctypes.byref(dp),
                              lse.data_ptr() if lse is not None else None, var,
                              _stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


def sdpa_math_plan(q, k, v, mask=None, is_causal=False, scale=None, out=None, probs=None,
                   variant="auto", out_shape=None, probs_shape=None):
    """Host-only validation + kernel-family choice.  Returns a dict; raises on error.

    Works on any tensors (CPU or meta shapes are fine): data pointers are only
    checked for NULL / alignment, never dereferenced.
    """
    lib = load_library()
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1]) if q.shape[-1] > 0 else 1.0
    if out is None:
        out = torch.empty(out_shape or (*q.shape[:3], v.shape[-1]), dtype=q.dtype)
    if probs is None:
        probs = torch.empty(probs_shape or (*q.shape[:3], k.shape[-2]), dtype=q.dtype)
    dq, dk, dv, do, dp = describe(q), describe(k), describe(v), describe(out), describe(probs)
    dm = describe(mask) if mask is not None else None
    plan = SdpaPlan()
    var = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    st = lib.sdpa_math_plan(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                            ctypes.byref(dm) if dm is not None else None, _mask_kind(mask),
                            int(bool(is_causal)), float(scale), ctypes.byref(do), ctypes.byref(dp),
                            var, ctypes.byref(plan))
    if st != SDPA_OK:
        _raise(lib, st)
    return {"variant": VARIANT_NAMES.get(plan.variant, plan.variant),
            "live_score_tiles": plan.live_score_tiles, "launches": plan.launches}


def sdpa_math_device_status(stream=None) -> None:
    lib = load_library()
    st = lib.sdpa_math_device_status(_stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


# Backward kernel families (sdpa_math_bwd_ex): "tc" = the tensor-core kernels.
BWD_VARIANTS = {"auto": 0, "simt": 1, "tc": 2}


def sdpa_math_bwd(q, k, v, probs, dout, dprobs, scale, dq, dk, dv, rowsum, stream=None,
                  variant: str = "auto") -> None:
    """Direct C-ABI backward on caller-allocated device tensors (raises on error).
    ``variant`` "auto" calls sdpa_math_bwd; "simt" / "tc" force a family through
    sdpa_math_bwd_ex."""
    lib = load_library()
    args = [describe(t) for t in (q, k, v, probs, dout)]
    dg = describe(dprobs) if dprobs is not None else None
    outs = [describe(t) for t in (dq, dk, dv)]
    common = [*(ctypes.byref(a) for a in args), ctypes.byref(dg) if dg is not None else None,
              float(scale), *(ctypes.byref(o) for o in outs), rowsum.data_ptr() if rowsum is not None else None]
    if variant == "auto":
        st = lib.sdpa_math_bwd(*common, _stream_handle(stream))
    else:
        code = BWD_VARIANTS[variant] if isinstance(variant, str) else int(variant)
        st = lib.sdpa_math_bwd_ex(*common, code, _stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


def sdpa_math_bwd_noalloc(q, k, v, probs, dout, dprobs, scale, dq, dk, dv, stream=None) -> None:
    """The C-ABI backward that allocates nothing and takes no row-sum buffer
    (for callers that cannot allocate device memory at call time); the
    library keeps the per-row sums in its own fixed device array, so at most
    SDPA_BWD_NOALLOC_MAX_ROWS query rows (B*Hq*Sq) per call.  Raises on error."""
    lib = load_library()
    args = [describe(t) for t in (q, k, v, probs, dout)]
    dg = describe(dprobs) if dprobs is not None else None
    outs = [describe(t) for t in (dq, dk, dv)]
    st = lib.sdpa_math_bwd_noalloc(*(ctypes.byref(a) for a in args), ctypes.byref(dg) if dg is not None else None,
                                   float(scale), *(ctypes.byref(o) for o in outs), _stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


def sdpa_math_backward(q, k, v, probs, dout, dprobs=None, scale: Optional[float] = None, stream=None,
                       variant: str = "auto"):
    """(dq, dk, dv) of the (O, P) forward for gradients dout (of O) and dprobs
    (of P, optional), given the forward's P; CUDA tensors through the C ABI.
    Allocates the outputs and the per-row workspace (B*Hq*Sq floats)."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1]) if q.shape[-1] > 0 else 1.0
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rowsum = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    sdpa_math_bwd(q, k, v, probs, dout, dprobs, scale, dq, dk, dv, rowsum, stream, variant)
    return dq, dk, dv


def sdpa_math_selftest_wait(stream=None) -> None:
    """Enqueue the bounded-wait self test (a wait that runs out after ~1 s)."""
    lib = load_library()
    st = lib.sdpa_math_selftest_wait(_stream_handle(stream))
    if st != SDPA_OK:
        _raise(lib, st)


def sdpa_math_last_error() -> str:
    return load_library().sdpa_math_last_error().decode(errors="replace")


def sdpa_math_abi_version() -> int:
    return int(load_library().sdpa_math_abi_version())


def empty_outputs(q, v, Skv, dtype=None):
    """O [B,Hq,Sq,Dv] and P [B,Hq,Sq,Skv] as two views of one allocation
    (one ``empty`` for both; P first, O after it on a 256-byte boundary)."""
    import torch
    B, Hq, Sq = q.shape[:3]
    Dv = v.shape[-1]
    dtype = dtype or q.dtype
    esz = torch.empty((), dtype=dtype).element_size()
    np_ = B * Hq * Sq * Skv
    no = B * Hq * Sq * Dv
    align = 256 // esz
    off = (np_ + align - 1) // align * align
    buf = torch.empty(off + no, dtype=dtype, device=q.device)
    P = buf[:np_].view(B, Hq, Sq, Skv)
    O = buf[off:off + no].view(B, Hq, Sq, Dv)
    return O, P


def prepare_mask(attn_mask, B: int, Hq: int, Sq: int, Skv: int, dtype):
    """A mask broadcastable to [B, Hq, Sq, Skv] (bool, or additive of any
    floating type) as the C ABI takes it: [1|B, 1|Hq, Sq, Skv] with unit
    innermost stride.  Broadcast query / key dimensions (a key-padding mask
    [B, 1, 1, Skv], say) are materialised; batch and head dimensions of extent
    1 stay broadcast; an additive mask of another floating type becomes fp32."""
    import torch
    if attn_mask is None:
        return None
    m = attn_mask
    if m.dtype != torch.bool and m.dtype not in (dtype, torch.float32):
        m = m.to(torch.float32)
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4:
        raise ValueError(f"attn_mask must have at most 4 dimensions, got {attn_mask.dim()}")
    mb = B if m.shape[0] != 1 else 1
    mh = Hq if m.shape[1] != 1 else 1
    m = m.expand(mb, mh, Sq, Skv)
    if m.stride(2) == 0 or m.stride(3) != 1:
        m = m.contiguous()
    return m


def sdpa_math(q, k, v, attn_mask=None, dropout_p: float = 0.0, is_causal: bool = False,
              scale: Optional[float] = None, variant: str = "auto", return_lse: bool = False,
              stream=None):
    """(O, P) = SDPA math forward on CUDA tensors, through the C ABI.

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv] (f32/f16/bf16, innermost
    stride 1); attn_mask bool (True keeps) or additive, broadcastable to
    [1|B, 1|Hq, Sq, Skv].  ``scale`` defaults to 1/sqrt(D).  dropout_p must be
    0: dropout is not part of this operation.  With ``return_lse`` the call
    also returns the fp32 natural-log LSE per row, [B,Hq,Sq].
    """
    import torch
    if dropout_p != 0.0:
        raise ValueError("dropout_p must be 0: dropout is not part of this operation")
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1]) if q.shape[-1] > 0 else 1.0
    mask = prepare_mask(attn_mask, q.shape[0], q.shape[1], q.shape[2], k.shape[-2], q.dtype)
    O, P = empty_outputs(q, v, k.shape[-2])
    lse = None
    if return_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    sdpa_math_fwd_ex(q, k, v, mask, _mask_kind(mask), is_causal, scale, O, P, lse,
                     variant, stream)
    if return_lse:
        return O, P, lse
    return O, P
