"""The device-side timeout path, exercised without faulting or hanging a GPU.

The kernels bound every wait for a staged tile (mbarrier try_wait polls) and,
on expiry, record FM_ERR_KERNEL_TIMEOUT in the plan's error word and leave
through an OR-vote barrier. fm_selftest_wait_timeout runs that wait and exit
on an mbarrier that nothing completes, with a short poll limit, beside a
group whose barrier does complete. The host must then read the timeout from
fm_plan_poll_error (once: reading clears it), the other group must have
finished, and the context must stay usable: a forward call right after it
matches the oracle and reports no error.
"""
from __future__ import annotations

import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import WORKLOADS, make_input
from tests.gpu_util import check_close, oracle_for, plan_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


# the kernels' own limits (2^kWaitLog2Polls, 2^kIdleLog2Polls polls)
KERNEL_LOG2_POLLS = {0: 18, 1: 22}


@pytest.mark.parametrize("kind", [0, 1], ids=["tile-wait", "producer-wait"])
def test_wait_runs_out_and_is_reported_then_the_context_still_works(kind):
    import torch

    w = WORKLOADS["tiny"]
    plan = plan_for(w)
    try:
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        s = torch.cuda.current_stream().cuda_stream
        times = {}
        for log2 in (4, 8, 12):
            if log2 > 4 and times[log2 - 4] * 16 > 2e6:
                pytest.skip(f"2^{log2 - 4} polls took {times[log2 - 4]:.0f} us; not growing the wait further")
            done, us = fb.fm_selftest_wait_timeout(plan, kind, log2, s)
            times[log2] = us
            assert done == 1, "the group whose barrier completed must finish"
            assert fb.fm_plan_poll_error(plan) == fb.FM_ERR_KERNEL_TIMEOUT
            assert fb.fm_plan_poll_error(plan) == fb.FM_OK  # reading cleared it
            x = make_input(w)
            check_close(run_gpu(w, x, plan=plan), oracle_for(w, x), w.out_dtype, f"forward after 2^{log2} polls")
            assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        per_poll = (times[12] - times[8]) / ((1 << 12) - (1 << 8))
        give_up = per_poll * (1 << KERNEL_LOG2_POLLS[kind]) / 1e6
        print(f"\nwait kind {kind}: {per_poll * 1e3:.1f} ns per poll; the kernels' limit gives up after "
              f"{give_up:.2f} s; times {times}")
        assert times[12] > times[4]
        # the poll time is the hardware's (3.8 us per blocking poll on GB300 so
        # far); the bound only rules out a limit far from a second
        assert 0.01 < give_up < 5.0, "the kernels' wait limit should be about a second"
    finally:
        fb.fm_plan_destroy(plan)


def test_poll_limit_and_kind_are_checked():
    plan = plan_for(WORKLOADS["tiny"])
    try:
        for kind, bad in ((0, -1), (0, 40), (1, -1), (1, 40), (2, 4), (-1, 4)):
            with pytest.raises(fb.FmError):
                fb.fm_selftest_wait_timeout(plan, kind, bad)
    finally:
        fb.fm_plan_destroy(plan)
