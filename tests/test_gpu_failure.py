"""The failure path every kernel relies on, exercised on the GPU without a
fault: a kernel waits on an mbarrier phase that nothing completes; its bounded
wait must give up after the library's limit, report through the device error
word, and leave the context usable for the next call (here a DIFF V1 forward
checked against the oracle)."""
import threading
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


def test_an_error_on_one_stream_stays_on_that_stream():
    """Each stream has its own error word: while the self-test's bounded wait
    runs out on stream A (about 2 s), DIFF V1 forwards on stream B run to
    parity and B's word reads 0 -- reading it synchronises B only, and A's
    give-up neither cuts B's waits short nor is reported to B."""
    bd = binding()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    s = inputs.V1Shape(1, 300, 2, 64, 4, "bf16")
    x = inputs.make_v1(s, seed=21)
    xd = to_dev(x)
    ref = oracle_v1(x, s.layer_index)
    torch.cuda.synchronize()
    res = {}

    def on_a():
        try:
            res["code"] = bd.selftest_wait_limit(sa)
        except Exception as e:  # noqa: BLE001  (reported below)
            res["exc"] = e

    th = threading.Thread(target=on_a)
    th.start()
    outs, words = [], []
    with torch.cuda.stream(sb):
        t0 = time.monotonic()
        while len(outs) < 4 or (th.is_alive() and time.monotonic() - t0 < 30.0):
            outs.append(run_v1(xd, s.layer_index))
            words.append(bd.stream_error(sb))
            if len(outs) >= 64:
                break
    th.join(60.0)
    assert not th.is_alive()
    assert "exc" not in res, res.get("exc")
    assert res["code"] & 1, res                  # A's own give-up, reported on A
    assert words == [0] * len(words), words      # never on B
    for y in outs:
        assert_parity(y, ref, "bf16")
    assert bd.device_error() == 0                # A's word was cleared by its reader
