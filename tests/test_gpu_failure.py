"""Failure detection on the GPU without faulting it.

The grouped GEMMs' (W4A4 and W4A16) and the router GEMM's waits are bounded.
With the test-only fault injection (NVFP4MOE_TEST_DROP_STAGE=n: the first
GEMM launch of the process never arms its pipeline stage n) the consumers'
waits run out: the kernel must report NVFP4_E_DEVICE_TIMEOUT in the status
word, drain its copies and MMAs, free its tensor memory and return -- and the
context must stay usable: the same call right after gives the oracle's
result.  The library reads the variable once per process, so every scenario
runs in a child process (failure_scenarios.py) with the variable set.
Routing errors are reported the same way (status word, no trap): see
test_gpu_gemm.py::test_gemm_bad_offsets_report_status and
test_gpu_swiglu_combine.py::test_combine_out_of_range_rows_report_status.
"""
import json
import os
import subprocess
import sys

import pytest

from gpu_helpers import cuda_or_skip

pytestmark = pytest.mark.gpu

SCRIPT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "failure_scenarios.py")
NVFP4_E_DEVICE_TIMEOUT = 7


def _run(scenario, mode, drop):
    cuda_or_skip()
    env = dict(os.environ, NVFP4MOE_TEST_DROP_STAGE=str(drop))
    r = subprocess.run([sys.executable, SCRIPT, scenario, mode], env=env, capture_output=True, text=True,
                       timeout=900)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert r.returncode == 0 and lines, "scenario %s %s failed:\n%s\n%s" % (scenario, mode, r.stdout, r.stderr[-4000:])
    res = json.loads(lines[-1])
    assert res["status_injected"] == NVFP4_E_DEVICE_TIMEOUT and res["status_after"] == 0
    assert res["elapsed_s"] < 30.0
    return res


@pytest.mark.parametrize("mode", ["w4a4", "w4a16", "w4a8"])
def test_gemm_bounded_wait_times_out_and_context_survives(mode):
    _run("gemm", mode, 0)


@pytest.mark.parametrize("drop", [0, 1])
def test_pair_gemm_bounded_wait_times_out_and_context_survives(drop):
    """The CTA-pair GEMM: both CTAs of every pair give up, meet at their final
    cluster barrier, free their tensor memory and return."""
    _run("gemm_pair", "w4a4", drop)


def test_router_gemm_bounded_wait_times_out_and_context_survives():
    _run("router", "w4a4", 0)


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
@pytest.mark.parametrize("drop", [0, 3])
def test_layer_bounded_wait_times_out_and_context_survives(mode, drop):
    """The whole layer (its kernels chained as programmatic dependents): a GEMM
    stage that is never armed -- the first one, or one inside the first ring
    lap -- ends in a reported timeout, the kernels after it still run and
    return, and the next layer call gives the oracle's result."""
    _run("layer", mode, drop)
