"""GPU parity of the two-pass conv_out head (the head.cu page's temporal-then-spatial split).

Pass 1 is the swapped tcgen05 engine in its centre-tap form writing one plane of G per spatial tap
(12 channels each); pass 2 is the stencil kernel (nine spatial taps in fp32, bias, clamp, one
rounding, 2x2 unpatchify).

* head_two_pass (G in bf16, the page's value path) against the oracle's two-pass restatement with
  G rounded to bf16: exactly on sparse {-1,0,1} data, where every G value and sum is representable;
  within the random-data tolerance otherwise; against the exact single-pass head by PSNR.
* head_split (G in fp32) against the oracle's single-pass head: exactly on {-2..2} integer data
  (every partial sum is an integer below 2^24), within the tolerance and PSNR on random data.
"""
import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.ssim import ssim_rgb
from tests.gpu_helpers import (PSNR_MIN, SSIM_MIN, assert_close, assert_exact, crops_3d, dev, host_values, psnr,
                               sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def run_two_pass(x, carry, L, kernel="head_two_pass"):
    N, D, H, W, C = x.shape
    d = x3.make_desc(3, N, C, 12, H, W, D=D, layout="NDHWC", dtype="bf16", act="clamp", unpatchify2x2=True,
                     kernel=kernel)
    conv = x3.Conv(d, dev(L.w), dev(L.b))
    assert conv.kernel_name == kernel
    y = conv(dev(x), None if carry is None else dev(carry))
    torch.cuda.synchronize()
    return host_values(y, "bf16"), conv


def to_rgb(y12_ndhwc):
    """[N, D, H, W, 12] -> [N, D, 2H, 2W, 3] by the oracle's unpatchify."""
    return oracle.unpatchify2x2(y12_ndhwc.transpose(0, 4, 1, 2, 3)).transpose(0, 2, 3, 4, 1)


SHAPES = [(2, 9, 140), (3, 5, 300), (1, 17, 33), (4, 1, 7), (2, 12, 254)]


@pytest.mark.parametrize("shape", SHAPES, ids=str)
@pytest.mark.parametrize("variant", ["sparse1", "random"])
def test_two_pass_head(variant, shape):
    D, H, W = shape
    x, carry, L = synth.head(D=D, H=H, W=W, variant=variant, seed=3600 + H + W)
    got, _ = run_two_pass(x, carry, L)
    ref = to_rgb(oracle.head_two_pass(x.vals, L.w.vals, L.b.vals, carry=carry.vals, layout="NDHWC"))
    assert got.shape == ref.shape == (1, D, 2 * H, 2 * W, 3)
    if variant == "sparse1":
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)
        exact = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp",
                                            layout="NDHWC"))
        assert psnr(got, exact) >= PSNR_MIN
        if min(2 * H, 2 * W) >= 11:
            assert ssim_rgb(got, exact) >= SSIM_MIN


def test_two_pass_head_without_carry_and_batch():
    x, _, L = synth.head(D=2, H=6, W=70, variant="random", seed=3690)
    xs = np.concatenate([x.vals, x.vals[:, ::-1]], axis=0)          # N = 2, second sequence reversed
    xt = synth.Tensor(*synth.to_storage(xs, "bf16"), "bf16")
    got, _ = run_two_pass(xt, None, L)
    ref = to_rgb(oracle.head_two_pass(xt.vals, L.w.vals, L.b.vals, layout="NDHWC"))
    assert_close(got, ref)


def test_two_pass_head_full_size_sampled():
    """4 x 352 x 624 latent frames, 256 channels: outputs at sampled positions, each from the
    oracle's two-pass head run on that position's own 3x3x3 window."""
    x, carry, L = synth.head(seed=3950)
    got, _ = run_two_pass(x, carry, L)
    assert got.shape == (1, 4, 704, 1248, 3)
    seq = np.concatenate([carry.vals, x.vals], axis=1)
    pos = sample_positions(4, 352, 624, 300, seed=77)
    cr = crops_3d(seq, pos)
    y = oracle.head_two_pass(cr[:, 2:3], L.w.vals, L.b.vals, carry=cr[:, 0:2], layout="NDHWC")[:, 0, 1, 1, :]
    ref = to_rgb(y[:, None, None, None, :])[:, 0]                   # [n, 2, 2, 3]
    g = np.stack([got[0, t, 2 * h:2 * h + 2, 2 * w:2 * w + 2] for (t, h, w) in pos])
    assert_close(g, ref)


@pytest.mark.parametrize("shape", SHAPES, ids=str)
@pytest.mark.parametrize("variant", ["int", "sparse1", "random"])
def test_split_head(variant, shape):
    D, H, W = shape
    x, carry, L = synth.head(D=D, H=H, W=W, variant=variant, seed=3700 + H + W)
    got, _ = run_two_pass(x, carry, L, kernel="head_split")
    ref = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp", layout="NDHWC"))
    assert got.shape == ref.shape
    if variant != "random":   # int: mostly clamped values; sparse1: small unclamped sums
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)
        assert psnr(got, ref) >= PSNR_MIN
        if min(2 * H, 2 * W) >= 11:
            assert ssim_rgb(got, ref) >= SSIM_MIN
        split = to_rgb(oracle.head_two_pass(x.vals, L.w.vals, L.b.vals, carry=carry.vals, round_g=False,
                                            layout="NDHWC"))
        assert_close(got, split)


def test_split_head_full_size_sampled():
    x, carry, L = synth.head(seed=3960)
    got, _ = run_two_pass(x, carry, L, kernel="head_split")
    assert got.shape == (1, 4, 704, 1248, 3)
    seq = np.concatenate([carry.vals, x.vals], axis=1)
    pos = sample_positions(4, 352, 624, 300, seed=78)
    cr = crops_3d(seq, pos)
    y = oracle.conv3d_causal(cr[:, 2:3], L.w.vals, L.b.vals, carry=cr[:, 0:2], act="clamp",
                             layout="NDHWC")[:, 0, 1, 1, :]
    ref = to_rgb(y[:, None, None, None, :])[:, 0]
    g = np.stack([got[0, t, 2 * h:2 * h + 2, 2 * w:2 * w + 2] for (t, h, w) in pos])
    assert_close(g, ref)


@pytest.mark.parametrize("kernel", ["head_split", "head_stencil", "auto"])
def test_head_full_size_decoded_quality(kernel):
    """All 4 decoded 704x1248 RGB frames of the full-size head against the oracle's head computed in
    full: PSNR and SSIM (the second quality metric) of the decoded output, plus the tolerance."""
    x, carry, L = synth.head(seed=3970)
    N, D, H, W, C = x.shape
    d = x3.make_desc(3, N, C, 12, H, W, D=D, act="clamp", unpatchify2x2=True, kernel=kernel)
    conv = x3.Conv(d, dev(L.w), dev(L.b))
    got = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    ref = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp", layout="NDHWC"))
    assert got.shape == ref.shape == (1, 4, 704, 1248, 3)
    assert_close(got, ref)
    assert psnr(got, ref) >= PSNR_MIN
    assert ssim_rgb(got, ref) >= SSIM_MIN


def run_head(x, carry, L, kernel):
    N, D, H, W, C = x.shape
    d = x3.make_desc(3, N, C, 12, H, W, D=D, layout="NDHWC", dtype="bf16", act="clamp", unpatchify2x2=True,
                     kernel=kernel)
    conv = x3.Conv(d, dev(L.w), dev(L.b))
    y = conv(dev(x), None if carry is None else dev(carry))
    torch.cuda.synchronize()
    return host_values(y, "bf16"), conv


@pytest.mark.parametrize("shape", SHAPES + [(2, 15, 29), (1, 28, 14), (2, 7, 31), (1, 6, 30), (2, 23, 61),
                                            (1, 14, 60)], ids=str)
@pytest.mark.parametrize("variant", ["int", "sparse1", "random"])
def test_stencil_head(variant, shape):
    """The head in one kernel with the spatial stencil in the epilogue: exact on integer data against
    the oracle's single-pass head, and bit for bit the split form's values (same fp32 sums in the same
    order) on random data; shapes around the 30-column strips and 8-row windows (a column past a
    strip, exactly one or two strips, heights that fill their last window exactly or by one row)."""
    D, H, W = shape
    x, carry, L = synth.head(D=D, H=H, W=W, variant=variant, seed=3800 + H + W)
    got, conv = run_head(x, carry, L, "head_stencil")
    assert conv.kernel_name == "igemm_tcgen05_sw128_head_stencil"
    ref = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp", layout="NDHWC"))
    assert got.shape == ref.shape
    if variant != "random":
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)
        assert psnr(got, ref) >= PSNR_MIN
        split, _ = run_head(x, carry, L, "head_split")
        assert np.array_equal(got, split)


# (D, H, W, N): plans whose CTAs each run several abutting windows down the strips, with runs that
# start mid-strip and runs that finish one strip and go on at the top of the next
RUN_SHAPES = [(2, 100, 300, 2), (4, 200, 600, 1), (3, 47, 1000, 1)]


@pytest.mark.parametrize("shape", RUN_SHAPES, ids=str)
@pytest.mark.parametrize("variant", ["int", "sparse1", "random"])
def test_stencil_head_window_runs(variant, shape):
    """The stencil head where each CTA runs consecutive windows of a strip that abut (no overlap): the
    output rows centred on a seam are finished from row sums carried from the window above, for every
    output frame. Exact on integer and sparse data against the oracle; on random data within the
    tolerance and bit for bit the split form (the carried sums keep the (i, j) order)."""
    D, H, W, N = shape
    x, carry, L = synth.head(D=D, H=H, W=W, N=N, variant=variant, seed=3900 + H + W)
    got, conv = run_head(x, carry, L, "head_stencil")
    g = x3.conv_plan_describe(conv.plan)
    assert conv.kernel_name == "igemm_tcgen05_sw128_head_stencil" and g["windows"] >= 2
    ref = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="clamp", layout="NDHWC"))
    assert got.shape == ref.shape
    if variant != "random":
        assert_exact(got, ref, "bf16")
        if variant == "sparse1":
            assert np.mean(np.abs(ref) < 1.0) > 0.0
    else:
        assert_close(got, ref)
        split, _ = run_head(x, carry, L, "head_split")
        assert np.array_equal(got, split)


def test_stencil_head_without_carry():
    x, _, L = synth.head(D=2, H=20, W=45, variant="int", seed=3890)
    got, _ = run_head(x, None, L, "head_stencil")
    ref = to_rgb(oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, act="clamp", layout="NDHWC"))
    assert_exact(got, ref, "bf16")
