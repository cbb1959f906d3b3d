"""Failure detection on the GPU without faulting it: a bounded device wait that runs out reports
X3_ERR_TIMEOUT through the device status word and leaves the context usable."""
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_exact, dev, host_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    assert x3.conv_device_status(1) == x3.X3_OK


def test_bounded_wait_times_out_and_context_survives():
    x3.conv_selftest_wait_timeout(50)                 # nothing ever arrives: the wait gives up after 50 ms
    assert x3.conv_device_status(0) == x3.X3_ERR_TIMEOUT
    assert "bounded device wait" in x3.conv_last_error()
    assert x3.conv_device_status(1) == x3.X3_ERR_TIMEOUT  # read and clear
    assert x3.conv_device_status(0) == x3.X3_OK
    # the context still runs convolutions correctly afterwards
    x, carry, L = synth.conv3d_single(C_in=32, C_out=32, D=1, H=4, W=20, variant="int", seed=6100)
    conv = x3.Conv(x3.make_desc(3, 1, 32, 32, 4, 20, D=1), dev(L.w), dev(L.b))
    got = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, layout="NDHWC")
    assert_exact(got, ref, "bf16")
    assert x3.conv_device_status(1) == x3.X3_OK


def test_selftest_rejects_bad_limits():
    for bad in (0, -1, 5000):
        with pytest.raises(x3.X3Error) as e:
            x3.conv_selftest_wait_timeout(bad)
        assert e.value.status == x3.X3_ERR_INVALID
