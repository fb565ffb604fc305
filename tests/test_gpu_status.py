"""The bounded-wait paths of the bf16 kernels, exercised without any fault.

The state kernel and the tcgen05 prologue wait on their own asynchronous
operand copies with a bounded number of polls (and, in the one-launch prefill,
the state pass on the prologue's publication flags). The test hook makes one of
them skip its first copy, so its wait runs out (and with it every wait on what
that copy would have produced): the kernel must record the timeout, exit (after
freeing its tensor memory), and leave the context usable; gdn_device_status
reports it once and then clears it."""
import pytest
import torch

from chunked_gated_deltanet_gb300 import gdn
from chunked_gated_deltanet_gb300 import workloads as wl
from helpers import Runner

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads", [2, 64], ids=["one_launch", "two_launches"])
@pytest.mark.parametrize("which", [1, 2], ids=["state_kernel", "prologue"])
def test_wait_timeout_is_reported_and_context_survives(cuda_device, which, heads):
    """2 heads run as one launch (chains beside the prologue, publication flags between them); 64 heads as a
    prologue kernel and a state kernel."""
    shape = wl.Shape(heads, heads, 128, 128, 64, wl.BF16)
    w = wl.Workload("timeout", shape, seed=41, session_lengths=[256])
    run = Runner(shape, w.session_tokens(0), w.conv_weights(), cuda_device)
    assert gdn.gdn_device_status() == gdn.GDN_OK
    victim, out = run.session(), run.new_out()
    gdn.gdn_debug_inject_wait_timeout(which, 2000)
    try:
        run.prefill(victim, 0, 256, out)
        status = gdn.gdn_device_status()
    finally:
        gdn.gdn_debug_inject_wait_timeout(False)
    assert status == gdn.GDN_ERR_TIMEOUT
    assert gdn.gdn_device_status() == gdn.GDN_OK          # reported once, then cleared
    # the context still works and gives the same result as before
    a, b = run.session(), run.session()
    oa, ob = run.new_out(), run.new_out()
    run.prefill(a, 0, 256, oa)
    run.prefill(b, 0, 256, ob)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(oa, ob) and torch.equal(a.S, b.S)
    assert torch.isfinite(oa).all()
