"""The bounded wait of the library's kernels, exercised without a fault: a
kernel waits, with the same limits, on an mbarrier phase that nothing
completes. The wait must give up by its limit (about one second, or a cap on
polls), and the device must stay usable: a dispatch and combine right after
it still match the oracle exactly."""
import pytest

import combine_quant_gb300 as cq
import gpu_harness as gh
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_device_stays_usable():
    gave_up, secs = cq.check_bounded_wait()
    assert gave_up == 1
    assert 0.01 < secs < 5.0, secs
    assert cq.read_combine_status() == 0  # the probe reports through its own word
    gh.full_parity(workloads.tiny(0, 2))
