"""CPU checks of the parity tolerance itself: an output formed the way the
operation forms it (P rounded to the dtype, O = P V from that rounded P, O
rounded) must sit inside the derived allowance, and a plainly wrong output
must not."""
import numpy as np
import pytest
import torch

from oracle import oracle_fwd
from parity_util import compare, o_allowance
from sdpa_forward_materialised_gb300 import workloads as W


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [True, False])
def test_rounded_p_output_is_inside_the_allowance(dtype, causal):
    q, k, v, _ = W.make_custom(40, 2, 4, 2, 96, 96, 64, dtype)
    O, P, _ = oracle_fwd(q, k, v, is_causal=causal, scale=0.125)
    td = q.dtype
    Pr = torch.from_numpy(P).to(td)                                   # P as returned
    vr = v.double().repeat_interleave(2, dim=1)
    Osim = torch.matmul(Pr.double(), vr).to(td)                       # O from rounded P
    compare(Pr, P, td, "P")
    stats = compare(Osim, O, td, "O", extra=o_allowance(P, v, 2, td))
    assert stats["max_abs"] > 0


def test_wrong_output_fails():
    q, k, v, _ = W.make_custom(41, 1, 2, 2, 64, 64, 64, "bf16")
    O, P, _ = oracle_fwd(q, k, v, is_causal=True, scale=0.125)
    bad = torch.from_numpy(O).to(torch.bfloat16).double()
    bad[0, 1, 10, 3] += 0.05
    with pytest.raises(AssertionError):
        compare(bad, O, torch.bfloat16, "O", extra=o_allowance(P, v, 1, torch.bfloat16))


def test_f16_is_held_to_the_plain_tolerance():
    """An f16 O error of 2.5e-3 at a large magnitude fails: f16 and f32 get no
    ulp or rounded-P allowance, only the plain max-abs bound."""
    q, k, v, _ = W.make_custom(42, 1, 2, 2, 64, 64, 64, "f16")
    O, P, _ = oracle_fwd(q, k, v, is_causal=True, scale=0.125)
    got = torch.from_numpy(O).to(torch.float16).double()
    i = np.unravel_index(np.argmax(np.abs(O)), O.shape)
    assert abs(O[i]) > 2.0
    got[i] = float(O[i]) + 2.5e-3  # exactly 2.5e-3 off
    with pytest.raises(AssertionError):
        compare(got, O, torch.float16, "O", extra=o_allowance(P, v, 1, torch.float16))
