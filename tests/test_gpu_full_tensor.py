"""Full-size parity over every output element, in the launch configurations bench.py times.

Every case builds its plans from ``bench.layer_descs()`` (the descriptors the benchmark runs) and
checks that their tiling is the one a fresh plan of that descriptor gets, with several strips and
windows, so the strip, window and frame seams of the timed kernels are all inside the comparison.

* Integer-valued data are compared bit for bit with the oracle: every fp32 partial sum is an exact
  integer below 2^24, so the GPU's summation order cannot change a value and only indexing, halo,
  padding, carries and the epilogue can. Where a premise of that (the size of the sums) depends on
  the drawn data, the test asserts it.
* Random data are compared over the full tensor within max|d| <= 1.5e-2 max|ref| and
  rms(d) <= 4e-3 rms(ref) (the tolerances of the causal-conv definition in FastVideo head.cu's header
  comment: all 27 taps in one fp32 accumulator, one rounding at the store).

Workloads (TAESD conv page: the 2D chain; FastVideo head.cu page: the causal decoder layers and the
conv_out head): the 16->16 64x64 conv, the TAESD-like 7-layer chain, the causal 256->256 4+2x88x156
layer, the two chained causal 128->128 layers at 4+2x352x624 with their carries, the causal 256->128
layer at 176x312 and the conv_out head 256->12 with clamp and 2x2 unpatchify.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_close, assert_exact, dev, host_values

pytestmark = pytest.mark.gpu

GEOM_KEYS = ("Wt", "P", "HR", "strips", "windows", "frames", "n_h", "n_w", "tiles", "grid", "m64", "s2", "stn")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def bench_conv(desc_kwargs, L):
    """A Conv for one of the benchmark's descriptors, after checking its tiling against a fresh plan of
    the same descriptor (the plan bench.py's workload makes) and that it spans several tiles."""
    conv = x3.Conv(x3.make_desc(**desc_kwargs), dev(L.w), dev(L.b))
    fresh = x3.conv_plan_create(x3.make_desc(**desc_kwargs))
    try:
        want = x3.conv_plan_describe(fresh)
    finally:
        x3.conv_plan_destroy(fresh)
    got = x3.conv_plan_describe(conv.plan)
    assert got == want
    geo = got.get("shadow", got)
    assert geo["tiles"] > geo.get("grid", 1) or geo["tiles"] >= 2, geo
    return conv


def check(got, ref, variant, dtype):
    if variant == "random":
        assert_close(got, ref)
    else:
        assert_exact(got, ref, dtype)


def rounded(y, dtype="bf16"):
    return oracle.round_to(y, dtype)[0]


@pytest.mark.parametrize("variant", ["int", "random"])
def test_conv16_64x64_full(variant):
    dd = bench.layer_descs()["conv16"]
    x, L = synth.conv2d_single(variant=variant, seed=5201)
    conv = bench_conv(dd, L)
    got = host_values(conv(dev(x)), "f16")
    torch.cuda.synchronize()
    check(got, oracle.conv2d(x.vals, L.w.vals, L.b.vals, act="relu"), variant, "f16")


@pytest.mark.parametrize("variant", ["int", "random"])
def test_causal_256_4x88x156_full(variant):
    dd = bench.layer_descs()["conv256"]
    x, carry, L = synth.conv3d_single(C_in=256, C_out=256, D=4, H=88, W=156, variant=variant, seed=5202)
    conv = bench_conv(dd, L)
    got = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    check(got, oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="none", layout="NDHWC"),
          variant, "bf16")


@pytest.mark.parametrize("variant", ["int", "random"])
def test_causal_256to128_4x176x312_full(variant):
    dd = bench.layer_descs()["l3"]
    x, carry, L = synth.conv3d_single(C_in=256, C_out=128, D=4, H=176, W=312, variant=variant, seed=5203)
    conv = bench_conv(dd, L)
    got = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    check(got, oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="none", layout="NDHWC"),
          variant, "bf16")


@pytest.mark.parametrize("variant", ["int", "random"])
def test_causal_stack_128_4x352x624_full(variant):
    """The two chained 128->128 layers through conv_stack_forward with their carries (the carry-update
    kernels run beside the layers), against the oracle layer by layer with each intermediate rounded
    to bf16 as the library stores it; the new carries are the last two frames of each layer's input."""
    descs = bench.layer_descs()["stack"]
    st = synth.conv3d_stack(variant=variant, seed=5204)
    convs = [bench_conv(dd, L) for dd, L in zip(descs, st["layers"])]
    cdev = [dev(c).contiguous() for c in st["carries"]]
    y = x3.ConvStack(convs)(dev(st["x"]), carries=cdev, carry_valid=True)
    torch.cuda.synchronize()
    got = host_values(y, "bf16")
    L1, L2 = st["layers"]
    c1, c2 = (c.vals for c in st["carries"])
    y1 = rounded(oracle.conv3d_causal(st["x"].vals, L1.w.vals, L1.b.vals, carry=c1, act="relu", layout="NDHWC"))
    if variant == "int":
        # premise of exactness for layer 2: |every partial sum| <= max|input| * max_co sum|w[co]| + max|b| < 2^24
        bound = max(np.abs(y1).max(), np.abs(c2).max()) * np.abs(L2.w.vals).reshape(128, -1).sum(1).max() \
            + np.abs(L2.b.vals).max()
        assert bound < 2 ** 24, bound
    ref = oracle.conv3d_causal(y1, L2.w.vals, L2.b.vals, carry=c2, act="relu", layout="NDHWC")
    check(got, ref, variant, "bf16")
    assert np.array_equal(host_values(cdev[0], "bf16"), st["x"].vals[:, 2:4])
    if variant == "int":
        assert np.array_equal(host_values(cdev[1], "bf16"), y1[:, 2:4])
    else:
        assert_close(host_values(cdev[1], "bf16"), y1[:, 2:4])


@pytest.mark.parametrize("variant", ["int", "sparse1", "random"])
def test_head_256to12_4x352x624_full(variant):
    """The conv_out head as the benchmark runs it (the default plan: the stencil head), clamp and 2x2
    unpatchify, all 4 x 704 x 1248 RGB values: exact on {-2..2} data (mostly clamped values) and on
    sparse {-1,0,1} weights (small unclamped sums), within the tolerance on random data."""
    dd = bench.layer_descs()["head"]
    x, carry, L = synth.head(variant=variant, seed=5205)
    conv = bench_conv(dd, L)
    assert conv.kernel_name == "igemm_tcgen05_sw128_head_stencil"
    got = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    y12 = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp", layout="NDHWC")
    ref = oracle.unpatchify2x2(y12.transpose(0, 4, 1, 2, 3)).transpose(0, 2, 3, 4, 1)
    assert got.shape == ref.shape == (1, 4, 704, 1248, 3)
    check(got, ref, variant, "bf16")
    if variant == "sparse1":
        assert 0.0 < np.mean(np.abs(ref) < 1.0)  # unclamped values are present


@pytest.mark.parametrize("variant", ["fewtaps", "random"])
def test_taesd_chain_full(variant):
    """The 7-layer TAESD-like chain through conv_stack_forward (channels-last between the layers,
    stride-2 phases), N=4 at 256x256, against the oracle layer by layer with f16 intermediates. The
    'fewtaps' weights (three +-1 per output channel, integer bias) keep every value of the chain an
    exact integer inside f16's range, so that comparison is bit for bit."""
    descs = bench.layer_descs()["taesd"]
    xt, layers = synth.taesd_chain(variant=variant, seed=5206)
    convs = [bench_conv(dd, L) for dd, L in zip(descs, layers)]
    got = host_values(x3.ConvStack(convs)(dev(xt)), "f16")
    torch.cuda.synchronize()
    y = xt.vals
    for L in layers[:-1]:
        y = rounded(oracle.conv2d(y, L.w.vals, L.b.vals, stride=L.stride, act="relu"), "f16")
    ref = oracle.conv2d(y, layers[-1].w.vals, layers[-1].b.vals, act="relu")
    assert got.shape == (4, 64, 128, 128)
    if variant == "fewtaps":
        assert np.all(np.isfinite(ref)) and np.abs(ref).max() < 65504
        assert np.count_nonzero(ref) > ref.size // 8
    check(got, ref, "int" if variant == "fewtaps" else variant, "f16")
