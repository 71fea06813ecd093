"""The failure path every kernel relies on, exercised on the GPU without a
fault: a kernel waits on an mbarrier phase that nothing completes; its bounded
wait must give up after the library's limit, report through the device error
word, and leave the context usable for the next call (here a DIFF V1 forward
checked against the oracle)."""
import time

import pytest
import torch

import oracle
from differential_attention_causal_gb300 import inputs
from test_gpu_parity import assert_parity, binding, built, oracle_v1, run_v1, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    bd = binding()
    t0 = time.monotonic()
    code = bd.selftest_wait_limit()
    elapsed = time.monotonic() - t0
    assert code & 1, code                      # the timeout bit (kErrWaitTimeout)
    assert 1.5 < elapsed < 30.0, elapsed       # the 2 s limit of global time, not a hang
    assert bd.last_launch_count() == 1
    assert bd.device_error() == 0              # the call cleared the word again
    # the next call runs normally: its waits are not cut short by a stale error bit
    s = inputs.V1Shape(2, 200, 2, 64, 3, "bf16")
    x = inputs.make_v1(s, seed=9)
    y = run_v1(to_dev(x), s.layer_index)
    assert bd.device_error() == 0
    assert_parity(y, oracle_v1(x, s.layer_index), "bf16")


def test_a_stale_error_word_is_cleared_before_the_self_test():
    bd = binding()
    bd.selftest_wait_limit()
    assert bd.selftest_wait_limit() & 1        # a second run reports its own give-up again
    assert bd.device_error() == 0
    torch.cuda.synchronize()
