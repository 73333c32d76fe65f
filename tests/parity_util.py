"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (max-abs, on both O and P): f32 1e-5, f16 2e-3, bf16 8e-3.

f32 and f16 are held to the plain max-abs bound on every element: both
dtypes can represent the results that closely (the f16 half-ulp is 1.95e-3
for magnitudes in [4, 8)).

bf16 cannot: its half-ulp at magnitudes in [4, 8) is 1.6e-2, twice the
bound, so a correctly rounded bf16 O can miss 8e-3.  For bf16 only, an
element may instead be off by one bf16 ulp at the reference's magnitude, and
for O also by sum_j half-ulp(P_ij) * |V_j|: the operation returns P in the
input dtype and O = P V is formed from that rounded P (as the math backend
does).  compare() counts the bf16 elements that needed this allowance and
prints the count with the plain max-abs error.
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

    f32 / f16: every element within the plain max-abs tolerance.  bf16: the
    allowance per element is max(tol, ulp(|ref|) + extra), ``extra`` being the
    propagated rounding of P for O (``o_allowance``), None for P; the count of
    elements beyond the plain tolerance is printed."""
    g = got.detach().double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    if g.size == 0:
        return {"max_abs": 0.0, "ulp_allowance_used": 0}
    assert not np.isnan(g).any(), f"{what}: NaN in GPU output (unwritten or bad)"
    err = np.abs(g - r)
    tol = TOL[dtype]
    if dtype == torch.bfloat16:
        allow = np.maximum(tol, ulp(r, dtype) + (0.0 if extra is None else extra))
    else:
        allow = np.full(err.shape, tol)
    bad = err > allow
    if bad.any():
        idx = np.unravel_index(np.argmax(err - allow), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements beyond tolerance; worst at {idx}: "
            f"got {g[idx]!r} ref {r[idx]!r} err {err[idx]:.3e} allow {allow[idx]:.3e}")
    used = int((err > tol).sum())
    if dtype == torch.bfloat16:
        print(f"[parity] {what}: max-abs {float(err.max()):.3e}, bf16 elements beyond {tol:g} "
              f"inside the ulp allowance: {used}")
    return {"max_abs": float(err.max()), "ulp_allowance_used": used}


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
