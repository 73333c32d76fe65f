"""CPU oracle for the materialised-probability SDPA forward (test infrastructure).

This package is test infrastructure.  Only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the product library never
does, and nothing here imports the product package.

``oracle_fwd`` widens the caller's tensors to float64 and runs the plain C
implementation in ``sdpa_oracle.c`` (textbook softmax in double precision).  The
operation follows FlagOS-OP PR #10 "feat: add sdpa_math operator": the SDPA math
backend returns (out, attn_probs) with causal and attn_mask mutually exclusive, a
bool mask meaning -inf masking, a fully masked row giving P = O = 0 and GQA
requiring Hq divisible by Hkv.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, hand-derived exact
rationals, brute force and an independent float64 library evaluation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsdpa_oracle.so")

MASK_NONE, MASK_BOOL, MASK_ADDITIVE = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP on) into ``oracle/_build``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
            lib.sdpa_oracle_fwd.restype = ctypes.c_int
            lib.sdpa_oracle_fwd.argtypes = [
                dp, dp, dp, dp, ctypes.c_int, i64, i64,
                i64, i64, i64, i64, i64, i64, i64,
                ctypes.c_int, ctypes.c_double, ctypes.POINTER(i64), i64,
                dp, dp, dp, ctypes.c_int]
            lib.sdpa_oracle_bwd.restype = ctypes.c_int
            lib.sdpa_oracle_bwd.argtypes = [
                dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, i64, i64,
                ctypes.c_double, dp, dp, dp, ctypes.c_int]
            lib.sdpa_oracle_max_threads.restype = ctypes.c_int
            lib.sdpa_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().sdpa_oracle_max_threads())


def _as_f64(x) -> np.ndarray:
    """Exact widening of a CPU tensor / array of any float or bool dtype to float64."""
    if hasattr(x, "detach"):  # torch tensor (fp16 / bf16 / fp32 / bool)
        x = x.detach().cpu()
        if x.dtype.is_floating_point:
            x = x.double()
        else:
            x = x.to(dtype=__import__("torch").float64)
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class OracleError(ValueError):
    pass


def oracle_fwd(q, k, v, attn_mask=None, is_causal: bool = False, scale=None,
               rows=None, nthreads: int = 1, mask_kind=None):
    """(O, P, lse) of the SDPA math forward, in float64.

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv]; attn_mask broadcastable as
    [1|B, 1|Hq, Sq, Skv] (bool: True keeps the key, False masks it with -inf;
    float: added to the scaled scores).  ``scale`` defaults to 1/sqrt(D).
    ``rows`` selects flattened rows ((b*Hq + h)*Sq + i); the outputs are then
    [nrows, Dv], [nrows, Skv], [nrows].  Without ``rows`` the outputs are
    [B,Hq,Sq,Dv], [B,Hq,Sq,Skv], [B,Hq,Sq].
    """
    lib = _load()
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    if qd.ndim != 4 or kd.ndim != 4 or vd.ndim != 4:
        raise OracleError("q, k, v must be rank 4")
    B, Hq, Sq, D = qd.shape
    Bk, Hkv, Skv, Dk = kd.shape
    Dv = vd.shape[3]
    if Bk != B or vd.shape[0] != B or vd.shape[1] != Hkv or vd.shape[2] != Skv or Dk != D:
        raise OracleError("q/k/v shapes disagree")
    if scale is None:
        scale = 1.0 / np.sqrt(D) if D > 0 else 1.0
    kind = MASK_NONE
    md = None
    mb = mh = 1
    if attn_mask is not None:
        is_bool = (getattr(attn_mask, "dtype", None) is not None
                   and str(attn_mask.dtype) in ("torch.bool", "bool"))
        kind = mask_kind if mask_kind is not None else (MASK_BOOL if is_bool else MASK_ADDITIVE)
        md = _as_f64(attn_mask)
        while md.ndim < 4:
            md = md[None]
        mb, mh = md.shape[0], md.shape[1]
        if md.shape[2] != Sq or md.shape[3] != Skv:
            raise OracleError("mask must be [1|B, 1|Hq, Sq, Skv]")
        md = np.ascontiguousarray(md)
    if rows is None:
        nrows = B * Hq * Sq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        nrows = rows_arr.size
    out = np.zeros((max(nrows, 0), Dv), dtype=np.float64)
    probs = np.zeros((max(nrows, 0), Skv), dtype=np.float64)
    lse = np.zeros((max(nrows, 0),), dtype=np.float64)
    dummy = np.zeros(1, dtype=np.float64)
    rc = lib.sdpa_oracle_fwd(
        _ptr(qd if qd.size else dummy), _ptr(kd if kd.size else dummy),
        _ptr(vd if vd.size else dummy), _ptr(md) if md is not None else None,
        kind, mb, mh, B, Hq, Hkv, Sq, Skv, D, Dv, int(bool(is_causal)), float(scale),
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        nrows, _ptr(out if out.size else dummy), _ptr(probs if probs.size else dummy),
        _ptr(lse if lse.size else dummy), int(nthreads))
    if rc != 0:
        raise OracleError(
            "oracle rejected the arguments (GQA indivisible, causal with a mask, "
            "bad mask broadcast or bad row id)")
    if rows is None:
        return (out.reshape(B, Hq, Sq, Dv), probs.reshape(B, Hq, Sq, Skv),
                lse.reshape(B, Hq, Sq))
    return out, probs, lse


def oracle_bwd(q, k, v, probs, dout, dprobs=None, scale=None, nthreads: int = 1):
    """(dq, dk, dv) in float64 for L = sum(O * dout) + sum(P * dprobs), given the
    forward's probability map ``probs`` [B,Hq,Sq,Skv] (see sdpa_oracle_bwd):
    dS = P * (dP - rowsum(P * dP)) with dP = dout V^T + dprobs; dq = scale dS K,
    dk = scale dS^T Q and dv = P^T dout, summed over each KV head's query heads."""
    lib = _load()
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    pd, god = _as_f64(probs), _as_f64(dout)
    B, Hq, Sq, D = qd.shape
    Hkv, Skv, Dv = kd.shape[1], kd.shape[2], vd.shape[3]
    if pd.shape != (B, Hq, Sq, Skv) or god.shape != (B, Hq, Sq, Dv):
        raise OracleError("probs / dout shapes disagree with q, k, v")
    gpd = None
    if dprobs is not None:
        gpd = _as_f64(dprobs)
        if gpd.shape != (B, Hq, Sq, Skv):
            raise OracleError("dprobs must be [B,Hq,Sq,Skv]")
    if scale is None:
        scale = 1.0 / np.sqrt(D) if D > 0 else 1.0
    dq = np.zeros((B, Hq, Sq, D), dtype=np.float64)
    dk = np.zeros((B, Hkv, Skv, D), dtype=np.float64)
    dv = np.zeros((B, Hkv, Skv, Dv), dtype=np.float64)
    dummy = np.zeros(1, dtype=np.float64)
    f = lambda a: _ptr(a if a.size else dummy)
    rc = lib.sdpa_oracle_bwd(f(qd), f(kd), f(vd), f(pd), f(god), _ptr(gpd) if gpd is not None else None,
                             B, Hq, Hkv, Sq, Skv, D, Dv, float(scale), f(dq), f(dk), f(dv), int(nthreads))
    if rc != 0:
        raise OracleError("oracle rejected the arguments (GQA indivisible or bad sizes)")
    return dq, dk, dv
