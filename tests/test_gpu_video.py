"""Pass-by-pass decoding of a long sequence (carries between passes) equals the oracle over the whole
sequence and one long pass on the GPU, and the device memory it needs does not grow with the sequence
length."""
import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from x3x3_convolution_gb300.video import PassDecoder
from tests.gpu_helpers import dev, host_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def _layers(D, H, W, seed):
    chans = [16, 32, 16]
    Ls = [synth.make_layer([seed, i], 3, ci, co, "bf16", act="relu" if i == 0 else "none", variant="int")
          for i, (ci, co) in enumerate(zip(chans[:-1], chans[1:]))]
    return Ls, [x3.Conv(x3.make_desc(3, 1, L.C_in, L.C_out, H, W, D=D, act=L.act), dev(L.w), dev(L.b)) for L in Ls]


def test_passes_equal_one_long_pass():
    T, D, H, W = 10, 4, 6, 40
    Ls, convs4 = _layers(D, H, W, 7100)
    _, convsT = _layers(T, H, W, 7100)
    x = synth.activation([7100, 0], (1, T, H, W, 16), "bf16", "int")
    want = host_values(x3.ConvStack(convsT)(dev(x)), "bf16")
    # the one long pass against the oracle run layer by layer over the whole sequence (zero history,
    # each intermediate rounded to bf16 as the library stores it; integer data: exact)
    ref = x.vals
    for L in Ls:
        ref = oracle.round_to(oracle.conv3d_causal(ref, L.w.vals, L.b.vals, act=L.act, layout="NDHWC"), "bf16")[0]
    assert np.array_equal(want, ref)
    dec = PassDecoder(convs4, D)
    got = dec.decode(x.torch("cpu").pin_memory())                  # passes of 4, 4 and 2 frames
    assert got.device.type == "cpu"
    assert np.array_equal(host_values(got, "bf16"), want)
    # a device-resident sequence gives the same frames
    dec2 = PassDecoder(convs4, D)
    assert np.array_equal(host_values(dec2.decode(dev(x)), "bf16"), want)


def test_peak_memory_does_not_grow_with_length():
    D, H, W = 4, 16, 64
    _, convs = _layers(D, H, W, 7200)
    peaks = []
    for T in (8, 32):
        x = torch.zeros((1, T, H, W, 16), dtype=torch.bfloat16).pin_memory()
        dec = PassDecoder(convs, D)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        dec.decode(x)
        peaks.append(torch.cuda.max_memory_allocated() - base)
        del dec
    assert peaks[1] <= peaks[0] * 1.05 + 4096
