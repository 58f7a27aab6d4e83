"""Failure detection on the GPU without a fault: a kernel whose one bounded wait can never
complete (nothing arrives at its barrier) gives up after its bound, records the timeout in the
library's device error word and ends by itself; csa2_check reports it once and clears it, and
the device keeps computing correct results afterwards.
"""
import time

import pytest

import compressed_sparse_attention_03_gb300 as csa2
from test_gpu_parity import check_index, make_state, run_index

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    return csa2.csa2_create()


def test_timeout_is_reported_once_and_the_device_keeps_working(handle):
    assert csa2.csa2_check(handle) == 0  # nothing pending from earlier tests
    t0 = time.perf_counter()
    csa2.csa2_selftest_timeout(handle)
    assert csa2.csa2_check(handle) == 8  # CSA2_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert waited < 5.0, f"the bounded wait took {waited:.2f} s"
    print(f"bounded wait gave up and was reported after {1e3 * waited:.1f} ms")
    assert csa2.csa2_check(handle) == 0  # cleared
    # a normal call afterwards: exact parity again
    x, cap = make_state(2, 1, [3001, 1000], seed=17)
    idx, top = run_index(handle, x, [3001, 1000], 1)
    check_index(idx, top, x, [3001, 1000])
    assert csa2.csa2_check(handle) == 0
