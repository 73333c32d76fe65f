"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out is reported through sdpa_math_device_status, and the context
stays usable afterwards.

The self test waits, through the tensor-core kernels' own bounded mbarrier
wait, on a barrier that nothing arrives at (no trap, no bad address, no
endless loop); the wait gives up after about one second.
"""
import math

import pytest
import torch

import sdpa_forward_materialised_gb300 as sm
from sdpa_forward_materialised_gb300 import workloads as W
from oracle import oracle_fwd
from parity_util import compare, o_allowance

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    sm.sdpa_math_device_status()  # start from a clean status word
    sm.sdpa_math_selftest_wait()
    with pytest.raises(sm.SdpaError) as ei:
        sm.sdpa_math_device_status()
    assert sm.STATUS[ei.value.status] == "SDPA_ERR_TIMEOUT", str(ei.value)
    assert "role 15" in str(ei.value)
    # the status word was cleared by the read
    sm.sdpa_math_device_status()


def test_context_usable_after_a_timeout():
    sm.sdpa_math_selftest_wait()
    with pytest.raises(sm.SdpaError):
        sm.sdpa_math_device_status()
    q, k, v, m = W.make_custom(7, 1, 2, 2, 136, 136, 64, "f16")
    scale = 1.0 / math.sqrt(64)
    O, P = sm.sdpa_math(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    sm.sdpa_math_device_status()
    Or, Pr, _ = oracle_fwd(q, k, v, None, is_causal=False, scale=scale)
    compare(P.cpu(), Pr, q.dtype, "P")
    compare(O.cpu(), Or, q.dtype, "O", extra=o_allowance(Pr, v, 1, q.dtype))
