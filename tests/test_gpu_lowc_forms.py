"""Edge cases of the low-channel forms of the channels-last engine, against the oracle bit for bit on
integer data and within the tolerances on random data:

* TN (positions as M = 128, the three horizontal taps x C_out in N, raster pitch 32, four raster rows
  per tile, 64-channel rows written by TMA stores): images narrower than one 30-column strip, exactly
  one strip, one column past a strip, heights that leave a partial last tile, one row, batches,
  several 64-channel input chunks with a partial last one, every padded output width 16..80;
* TK (8 input channels, two taps per K step);
* both in banded mode at a band's top, middle and bottom.
The definition is the TAESD conv page's taesd_conv3x3_impl (pad-1 3x3 cross-correlation, bias-
initialised fp32 accumulator, ReLU, one rounding at the store)."""
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_close, assert_exact, dev, host_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


CASES = [
    # (N, C_in, C_out, H, W)
    (1, 64, 64, 4, 29),     # narrower than a strip, exactly one tile of rows
    (2, 64, 64, 5, 30),     # exactly one strip, a second (partial) tile of rows
    (1, 64, 64, 9, 31),     # one column past a strip
    (3, 16, 32, 1, 90),     # one row, three strips, a batch
    (1, 72, 64, 13, 60),    # two input chunks, the second partial (8 channels)
    (1, 200, 48, 6, 33),    # four input chunks
    (2, 8, 64, 11, 47),     # TK
    (1, 8, 16, 3, 2),       # TK, tiny
    (1, 8, 80, 6, 61),      # TK, 80 output channels
    (2, 32, 80, 7, 35),     # TN, N = 240
    (1, 64, 16, 17, 64),    # TN, N = 48
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", CASES, ids=str)
def test_lowc_forms(case, variant, dtype):
    N, Ci, Co, H, W = case
    key = 7300 + sum(case)
    x = synth.activation([key, 0], (N, H, W, Ci), dtype, variant, ("uniform", -1.0, 1.0))
    L = synth.make_layer([key], 2, Ci, Co, dtype, act="relu", variant=variant)
    conv = x3.Conv(x3.make_desc(2, N, Ci, Co, H, W, layout="NHWC", dtype=dtype, act="relu"), dev(L.w), dev(L.b))
    g = x3.conv_plan_describe(conv.plan)
    assert g["tn"] == 1 or Ci * Co > 128 * 48, g
    got = host_values(conv(dev(x)), dtype)
    torch.cuda.synchronize()
    ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, act="relu", layout="NHWC")
    if variant == "int":
        assert_exact(got, ref, dtype)
    else:
        assert_close(got, ref)


@pytest.mark.parametrize("Ci", [8, 64])
def test_lowc_forms_banded(Ci):
    """TN / TK layers in banded mode: bands of 5, 9 and the rest of 23 rows, concatenated, equal the
    whole plane, which equals the oracle (integer data)."""
    N, Co, H, W = 2, 64, 23, 70
    x = synth.activation([7400, Ci], (N, H, W, Ci), "f16", "int")
    L = synth.make_layer([7400, Ci], 2, Ci, Co, "f16", act="relu", variant="int")
    base = dict(dims=2, N=N, C_in=Ci, C_out=Co, W=W, layout="NHWC", dtype="f16", act="relu")
    full = x3.Conv(x3.make_desc(H=H, **base), dev(L.w), dev(L.b))
    assert x3.conv_plan_describe(full.plan)["tk"] == (Ci == 8)
    xd = dev(x)
    y = full(xd)
    parts = []
    for lo, rows in [(0, 5), (5, 9), (14, 9)]:
        a, b = x3.band_input_rows(lo, rows, H)
        c = x3.Conv(x3.make_desc(H=b - a, band_lo=lo, band_rows=rows, H_global=H, **base), dev(L.w), dev(L.b))
        parts.append(c(xd[:, a:b].contiguous()))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), y)
    ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, act="relu", layout="NHWC")
    assert_exact(host_values(y, "f16"), ref, "f16")
