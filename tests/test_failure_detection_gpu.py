"""Device-side failure detection without a GPU fault: a bounded wait made to run out on
purpose reports LIZARD_ERR_TIMEOUT through the workspace's status word, the word is
cleared by reading it, and the context stays usable for normal calls afterwards."""
import numpy as np
import pytest
import torch

import hybrid_gated_linear_gb300 as lz
import oracle
import synth
from gpu_util import NAMES, TOL, gpu_fwd, rel_l2

pytestmark = pytest.mark.gpu

TIMEOUT = 4  # LIZARD_ERR_TIMEOUT


@pytest.mark.parametrize("cycles", [1, 200_000])
def test_bounded_wait_runs_out_and_is_reported(cycles):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lz.lizard_selftest_wait_timeout(ws, cycles)
    assert lz.lizard_last_launch_count() == 1
    assert lz.lizard_check_device_errors(ws) == TIMEOUT
    assert lz.lizard_check_device_errors(ws) == 0  # read once, then cleared


def test_normal_call_after_a_timeout():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lz.lizard_selftest_wait_timeout(ws, 100_000)
    assert lz.lizard_check_device_errors(ws) == TIMEOUT
    x = synth.make_fwd_inputs(1, 2, 200, 128, 128, 4, "bf16", "plain", seed=5)
    y, _ = gpu_fwd(x, 64, "bf16")  # asserts its own status word is 0
    ref = oracle.fwd(*(x[n] for n in NAMES), W=64)
    assert rel_l2(y, ref["y"]) <= TOL["bf16"]


def test_selftest_rejects_bad_arguments():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lz.LizardError) as e:
        lz.lizard_selftest_wait_timeout(ws, 0)
    assert e.value.status == 1
    with pytest.raises(lz.LizardError) as e:
        lz.lizard_selftest_wait_timeout(ws[:128], 1000)
    assert e.value.status == 6
