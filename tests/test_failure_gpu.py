"""Failure detection on the GPU without a GPU fault: every wait in the library's kernels is
bounded and, when it runs out, sets the device error word and lets the kernel return. A
self-test kernel waits on an mbarrier that nothing arrives on; the host reads the error
through gdn_check_device_error, and the context stays usable for the next call."""
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs

from helpers import TOL, cuda_inputs, oracle_fwd, rel

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
    gdn.gdn_selftest_wait_timeout(1024)
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_ERR_INTERNAL
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK  # read and cleared
    host = make_inputs(WORKLOADS["tiny_fwd"].with_(T=64, h0_std=0.3))
    out, h = gdn.gdn_recurrent(*[cuda_inputs(host)[n] for n in ("q", "k", "v", "g", "beta", "h0")])
    o_ref, h_ref = oracle_fwd(host)
    assert rel(out, o_ref) <= TOL["f32"] and rel(h, h_ref) <= TOL["f32"]
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK


def test_waits_after_a_timeout_give_up_early():
    """Once a wait has timed out (error word set), the kernels' later waits give up after
    about 4096 tries instead of running their full count of 4194304: the self-test's four
    later waits together take a few times the cycles of its first 4096-try wait, where
    four full waits would take about a thousand times as many."""
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_OK
    cycles = torch.zeros(3, dtype=torch.int64, device="cuda")
    gdn.gdn_selftest_wait_timeout(4096, cycles=cycles)
    first, later, counter = (int(x) for x in cycles.cpu())
    assert gdn.gdn_check_device_error() == gdn.binding.GDN_ERR_INTERNAL
    print(f"first wait {first} cycles, four later waits {later} cycles, counter wait {counter} cycles")
    assert first > 0 and later > 0
    assert later < 4 * 4 * first, (first, later)
    # the cross-CTA counter wait ran out (it never saw the counter raised) and reported it
    assert counter > 0


def test_selftest_rejects_unbounded_requests():
    with pytest.raises(gdn.GdnError):
        gdn.gdn_selftest_wait_timeout(0)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_selftest_wait_timeout(1 << 20)
