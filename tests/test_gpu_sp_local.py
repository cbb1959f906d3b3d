"""The row-band decode of x3x3_convolution_gb300.sp with the library's banded kernels, three ranks
emulated in one process on cuda:0 (halo rows copied between the bands): two passes of a causal stack
(two 128->128 layers with ReLU, then the conv_out head 128->12 with clamp and 2x2 unpatchify) with
per-band histories must equal the whole-plane decode (conv_stack_forward with carries, then the head)
bit for bit."""
import pytest
import torch

import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import sp, synth
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def test_local_band_decode_with_banded_kernels():
    D, H, W = 2, 45, 70
    specs = [dict(dims=3, N=1, C_in=128, C_out=128, D=D, H=H, W=W, act="relu"),
             dict(dims=3, N=1, C_in=128, C_out=128, D=D, H=H, W=W, act="relu"),
             dict(dims=3, N=1, C_in=128, C_out=12, D=D, H=H, W=W, act="clamp", unpatchify2x2=True)]
    Ls = [synth.make_layer([9200, i], 3, s["C_in"], s["C_out"], "bf16", act=s["act"]) for i, s in enumerate(specs)]
    xs = [synth.activation([9200, 10 + p], (1, D, H, W, 128), "bf16", "random", ("normal", 1.0)) for p in range(2)]
    # whole plane: the two layers through conv_stack_forward with carries, then the head with its carry
    full = [x3.Conv(x3.make_desc(**s), dev(L.w), dev(L.b)) for s, L in zip(specs, Ls)]
    stack = x3.ConvStack(full[:2])
    c_full = [torch.zeros((1, 2, H, W, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    want = []
    for p, x in enumerate(xs):
        xd = dev(x)
        mid = stack(xd, carries=c_full[:2], carry_valid=p > 0)
        want.append(full[2](mid, c_full[2] if p > 0 else None))
        c_full[2].copy_(torch.cat([c_full[2], mid], dim=1)[:, -2:] if p > 0 else mid[:, -2:])
    # three bands, each layer a banded Conv of the same weights
    world = 3
    bands = sp.LocalBands(H, row_axis=2, world=world)
    runs, carries = [], []
    for lo, rows in bands.bands:
        a, b = sp.halo_rows(lo, rows, H)
        convs = [sp.banded_conv(lambda d, L=L: x3.Conv(d, dev(L.w), dev(L.b)), s, lo, rows, H) for s, L in zip(specs, Ls)]
        runs.append([lambda inp, hist, c=c: c(inp, hist) for c in convs])
        carries.append([torch.zeros((1, 2, b - a, W, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3)])
    for p, x in enumerate(xs):
        parts = sp.decode_bands_local(runs, dev(x), carries, p > 0, bands)
        got = torch.cat(parts, dim=2)
        torch.cuda.synchronize()
        assert got.shape == want[p].shape == (1, D, 2 * H, 2 * W, 3)
        assert torch.equal(got, want[p])
