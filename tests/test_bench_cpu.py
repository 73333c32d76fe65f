"""bench.py's host-side paths that need no GPU: the reference (oracle) arm of
the forward and of the backward, their JSON lines, and the backward's byte
count and kernel-family rule."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sdpa_forward_materialised_gb300 import workloads as W  # noqa: E402


def _run(argv):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(argv)
    assert rc == 0
    return json.loads(buf.getvalue().strip().splitlines()[-1])


def test_reference_arm_forward_line():
    line = _run(["--impl", "reference", "--config", "tiny_f32", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.2"])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_backward_line():
    line = _run(["--impl", "reference", "--pass", "bwd", "--config", "tiny_f32", "--steps", "1", "--warmup", "3"])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC_BWD
    assert line["config"] == {"workload": "tiny_f32", "pass": "bwd"}
    assert line["higher_is_better"] is False and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and "groups" in line["cpu_baseline"]["sample"]


def test_backward_bytes_and_family():
    w = W.PREFILL_2K_D128
    rows = w.B * w.Hq * w.Sq
    # q, dout, dq rows; k, v, dk, dv rows; P and dprobs; fp32 row sums
    expect = 2 * (3 * rows * w.D + 4 * w.B * w.Hkv * w.Skv * w.D + 2 * rows * w.Skv) + 4 * rows
    assert bench.bwd_bytes(w) == expect
    assert bench.bwd_tc_eligible(w) and bench.bwd_tc_eligible(W.GQA_1K_D128)
    assert not bench.bwd_tc_eligible(W.TINY)        # fp32
    assert not bench.bwd_tc_eligible(W.TAIL100)     # 100 keys: P rows not on 16-byte boundaries
