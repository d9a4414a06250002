"""The bounded-wait give-up path on the GPU, without a fault: a self-test
kernel waits on an mbarrier that nothing completes; the wait runs out after
about 2 s and sets the library's status word; ssm_check_device_status reports
SSM_ERR_TIMEOUT once and clears it; the context stays usable and the next
scan is correct."""
import time

import pytest

from gpu_helpers import TOL, compare_all, gpu_fwd_bwd, oracle_fwd_bwd, to_dev
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_reports_timeout():
    s6.check_device_status()  # start clean
    t0 = time.perf_counter()
    s6.selftest_wait_timeout()
    with pytest.raises(s6.SSMError) as err:
        s6.check_device_status()
    waited = time.perf_counter() - t0
    assert "SSM_ERR_TIMEOUT" in str(err.value)
    assert 0.5 < waited < 30.0
    s6.check_device_status()  # the bit was cleared
    # the context is still usable: a scan right after is correct
    x = inputs.make_inputs(2, 100, 64, 16, "f32", seed=3, h0_std=0.5, with_dh_last=True)
    got = gpu_fwd_bwd(to_dev(x), dh_last=to_dev(x)["dh_last"])
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(got, ref, TOL["f32"])
