"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (max-abs, on both O and P): f32 1e-5, f16 2e-3, bf16 8e-3.  Where
the output dtype cannot represent the exact value that closely (bf16 values of
magnitude >= 4 have a half-ulp of 1.6e-2), an element may instead be off by at
most one ulp of the dtype at the reference's magnitude.  For O that allowance
also carries the rounding of P: the operation returns P in the input dtype and
O = P V is formed from that rounded P (as the math backend does), so O may
additionally differ from the exact fp64 value by sum_j half-ulp(P_ij) * |V_j|.
The number of elements that needed an allowance beyond the plain tolerance
is reported.
"""
import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 8e-3}
MANT = {torch.float32: 23, torch.float16: 10, torch.bfloat16: 7}
MIN_EXP = {torch.float32: -126, torch.float16: -14, torch.bfloat16: -126}


def ulp(ref: np.ndarray, dtype) -> np.ndarray:
    """One ulp of ``dtype`` at |ref| (the subnormal spacing below the normal range)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, MIN_EXP[dtype])
    return np.ldexp(1.0, (e - MANT[dtype]).astype(np.int64))


def p_rounding_bound(p_ref: np.ndarray, v_rows: np.ndarray, dtype) -> np.ndarray:
    """Bound on |O - O_exact| caused by rounding P to ``dtype`` before P V:
    sum_j (half an ulp of P[i,j]) * |V[j,:]|.  ``p_ref`` is [..., Skv] and
    ``v_rows`` the matching [..., Skv, Dv] values (already head-mapped)."""
    half = 0.5 * ulp(p_ref, dtype) * (p_ref != 0)
    return np.einsum("...j,...je->...e", half, np.abs(v_rows))


def o_allowance(p_ref: np.ndarray, v, group: int, dtype, rows=None, Hq=None, Sq=None) -> np.ndarray:
    """Per-element extra allowance for O (see p_rounding_bound).  Either full
    [B,Hq,Sq,Skv] references, or flattened ``rows`` with their (Hq, Sq)."""
    vn = (v.double().numpy() if torch.is_tensor(v) else np.asarray(v, np.float64))
    if rows is None:
        vr = np.repeat(vn, group, axis=1)                    # [B,Hq,Skv,Dv]
        return p_rounding_bound(p_ref, vr[:, :, None, :, :], dtype)
    b = rows // (Hq * Sq)
    h = (rows // Sq) % Hq
    vr = vn[b, h // group]                                   # [n,Skv,Dv]
    return p_rounding_bound(p_ref, vr, dtype)


def compare(got, ref, dtype, what="", extra=None):
    """Element-wise check; returns a stats dict, raises AssertionError on failure.

    The allowance per element is max(tol, ulp(|ref|) + extra): ``extra`` is
    the propagated rounding of P for O (``o_allowance``), None for P."""
    g = got.detach().double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    if g.size == 0:
        return {"max_abs": 0.0, "ulp_allowance_used": 0}
    assert not np.isnan(g).any(), f"{what}: NaN in GPU output (unwritten or bad)"
    err = np.abs(g - r)
    tol = TOL[dtype]
    allow = np.maximum(tol, ulp(r, dtype) + (0.0 if extra is None else extra))
    bad = err > allow
    if bad.any():
        idx = np.unravel_index(np.argmax(err - allow), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements beyond tolerance; worst at {idx}: "
            f"got {g[idx]!r} ref {r[idx]!r} err {err[idx]:.3e} allow {allow[idx]:.3e}")
    return {"max_abs": float(err.max()), "ulp_allowance_used": int((err > tol).sum())}


def row_sum_bound(dtype, skv: int) -> float:
    """Bound on |sum_j P[i,j] - 1| for P rounded to ``dtype`` from an exactly
    normalised fp32 row: half an ulp relative per element, plus subnormal
    spacing per element, plus fp32 slack."""
    sub = 2.0 ** (MIN_EXP[dtype] - MANT[dtype] - 1)
    return 2.0 ** (-MANT[dtype] - 1) + skv * sub + 1e-5


def sample_rows(B, Hq, Sq, n_random=256, seed=0):
    """Flattened row ids ((b*Hq + h)*Sq + i): tile-edge rows of a few heads
    plus random rows."""
    total = B * Hq * Sq
    rng = np.random.default_rng(seed)
    picks = set()
    edge_i = sorted({0, 1, Sq - 1} | {i for t in range(0, Sq, 128) for i in (t, t + 127) if i < Sq}
                    | {i for t in range(0, Sq, 64) for i in (t, t + 63) if i < Sq})
    for b in {0, B - 1}:
        for h in {0, Hq - 1, Hq // 2}:
            for i in edge_i:
                picks.add((b * Hq + h) * Sq + i)
    picks.update(rng.choice(total, size=min(n_random, total), replace=False).tolist())
    return np.array(sorted(picks), dtype=np.int64)
