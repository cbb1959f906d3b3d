"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Integer-valued inputs ({-2..2}) must match bit for bit (every fp32 partial sum is exact, so only
indexing, halo, padding, carry and epilogue can differ); random inputs must meet the relative
max / rms tolerances. Sizes span several tiles and a ragged tail; both the tcgen05 kernel and the
direct kernel are checked.
"""
import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.ssim import ssim_rgb
from tests.gpu_helpers import (assert_close, assert_exact, dev, host_values, oracle_sampled_3d, psnr,
                               sample_positions, PSNR_MIN, SSIM_MIN)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def run2d(x, L, layout="NCHW", kernel="auto", expect=None):
    N, C, H, W = x.shape if layout == "NCHW" else (x.shape[0], x.shape[3], x.shape[1], x.shape[2])
    d = x3.make_desc(2, N, C, L.C_out, H, W, stride=L.stride, layout=layout, dtype=x.dtype, act=L.act,
                     has_bias=L.b is not None, kernel=kernel)
    conv = x3.Conv(d, dev(L.w), None if L.b is None else dev(L.b))
    if expect:
        assert conv.kernel_name == expect, conv.kernel_name
    y = conv(dev(x))
    torch.cuda.synchronize()
    return host_values(y, x.dtype), conv


def oracle2d(x, L, layout="NCHW"):
    return oracle.conv2d(x.vals, L.w.vals, None if L.b is None else L.b.vals, stride=L.stride, act=L.act,
                         layout=layout)


# ------------------------------------------------------------------ 2D

CASES_2D = [
    # (N, C_in, C_out, H, W, stride, act)
    (1, 16, 16, 64, 64, 1, "relu"),      # the 16->16 64x64 single conv
    (2, 3, 64, 40, 264, 1, "relu"),      # 3-channel input, ragged width (264 = 2*128 + 8)
    (1, 64, 64, 37, 136, 1, "relu"),     # ragged height and width
    (2, 64, 48, 16, 64, 1, "none"),      # C_out not a multiple of the N tile
    (1, 24, 16, 9, 8, 1, "relu"),        # C_in not a multiple of the channel chunk
    (1, 1, 16, 1, 8, 1, "none"),         # a single row
    (2, 64, 64, 34, 70, 2, "relu"),      # stride 2, width not a multiple of 8 (direct kernel)
    (2, 64, 64, 34, 72, 2, "relu"),      # stride 2 on the tensor cores (phase planes)
    (1, 16, 32, 33, 136, 2, "none"),     # stride 2, odd height, ragged output tile
    (1, 3, 64, 9, 264, 2, "relu"),       # stride 2, 3 input channels
]


@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", CASES_2D, ids=lambda c: "x".join(map(str, c[:6])))
@pytest.mark.parametrize("kernel", ["auto", "direct"])
def test_conv2d_nchw(case, variant, kernel):
    N, Ci, Co, H, W, s, act = case
    x, L = synth.conv2d_single(N=N, C=Ci, C_out=Co, H=H, W=W, stride=s, act=act, variant=variant,
                               seed=2000 + sum(case[:6]))
    got, conv = run2d(x, L, kernel=kernel)
    if kernel == "auto" and W % 8 == 0:
        assert conv.kernel_name.startswith("igemm_tcgen05")
    ref = oracle2d(x, L)
    if variant == "int":
        assert_exact(got, ref, "f16")
    else:
        assert_close(got, ref)


NHWC_CASES = [(2, 16, 32, 20, 150, 1, "relu"), (1, 64, 64, 9, 300, 1, "none"), (1, 8, 16, 3, 5, 1, "none"),
              (2, 64, 64, 34, 72, 2, "relu"), (1, 40, 24, 17, 33, 2, "none"), (2, 64, 128, 33, 97, 1, "relu"),
              (1, 128, 64, 12, 130, 1, "relu"),
              # positions-as-M form (horizontal taps in N): 80 channels (N = 240), 24 (padded to 32),
              # 8 (padded to 16), a partial last input chunk (136 = 2 x 64 + 8), one-column images
              (1, 64, 80, 19, 301, 1, "relu"), (2, 24, 24, 11, 40, 1, "none"), (1, 64, 8, 5, 260, 1, "relu"),
              (1, 136, 32, 7, 45, 1, "none"), (3, 16, 16, 6, 1, 1, "relu"),
              # 64 channels: each raster row leaves by one TMA store, clipped at a ragged right edge
              (2, 32, 64, 7, 61, 1, "relu"), (1, 32, 48, 9, 70, 1, "clamp"),
              # 8 input channels: two taps per K step (five MMAs), 64 and 24 output channels
              (4, 8, 64, 37, 95, 1, "relu"), (1, 8, 24, 9, 31, 1, "none")]


@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", NHWC_CASES, ids=str)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("form", ["auto", "m64"])
def test_conv2d_nhwc(case, variant, dtype, form, monkeypatch):
    """Channels-last 2D layers on the swapped engine: stride 1 with at most 80 output channels in the
    positions-as-M form with the horizontal taps in N (or, with X3CONV_TN=0, the M = 64 form for at
    most 64 output channels, weights resident when they fit), the 128-row form, and stride 2 from the
    four input phases."""
    if form == "m64":
        monkeypatch.setenv("X3CONV_TN", "0")
    N, Ci, Co, H, W, s, act = case
    key = 2100 + sum(case[:6])
    x = synth.activation([key, 0], (N, H, W, Ci), dtype, variant, ("uniform", -1.0, 1.0))
    L = synth.make_layer([key], 2, Ci, Co, dtype, stride=s, act=act, variant=variant)
    got, conv = run2d(x, L, layout="NHWC")
    g = x3.conv_plan_describe(conv.plan)
    assert g["kernel"] == "igemm_tcgen05_sw128" and g["s2"] == (s == 2)
    if form == "auto" and s == 1 and Co <= 80 and not (Ci > 128 and Co > 32):
        assert g["tn"] == 1 and g["tk"] == (Ci == 8)
    elif form == "m64":
        assert g["tn"] == 0 and g["m64"] == (Co <= 64 and Ci <= 64)
    ref = oracle2d(x, L, layout="NHWC")
    if variant == "int":
        assert_exact(got, ref, dtype)
    else:
        assert_close(got, ref)


@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", [(4, 64, 64, 64, 64, "relu"), (1, 64, 64, 33, 97, "none"),
                                  (2, 8, 32, 17, 255, "relu"), (1, 64, 128, 20, 66, "relu"),
                                  (1, 96, 64, 15, 40, "none"), (1, 136, 200, 9, 31, "none")], ids=str)
@pytest.mark.parametrize("form", ["phases", "raster"])
def test_conv2d_nhwc_stride2_forms(case, variant, form, monkeypatch):
    """Stride 2 on the channels-last engine in both forms: from the four input phases (element-strided
    boxes; the default), and with X3CONV_S2=0 as the stride-1 raster with even positions kept. Odd
    input sizes put the bottom and right taps in the zero padding; C_out > 64 takes the 128-row form
    and C_in > 64 two chunks per phase."""
    monkeypatch.setenv("X3CONV_S2", "1" if form == "phases" else "0")
    N, Ci, Co, H, W, act = case
    key = 2700 + sum(case[:5])
    x = synth.activation([key, 0], (N, H, W, Ci), "bf16", variant, ("uniform", -1.0, 1.0))
    L = synth.make_layer([key], 2, Ci, Co, "bf16", stride=2, act=act, variant=variant)
    got, conv = run2d(x, L, layout="NHWC")
    g = x3.conv_plan_describe(conv.plan)
    assert (g["s2"], g["sub2"]) == ((1, 0) if form == "phases" else (0, 1))
    ref = oracle2d(x, L, layout="NHWC")
    if variant == "int":
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)


# ------------------------------------------------------------------ 3D causal

def run3d(x, carry, L, kernel="auto", unpatch=False, dtype="bf16"):
    N, D, H, W, C = x.shape
    d = x3.make_desc(3, N, C, L.C_out, H, W, D=D, layout="NDHWC", dtype=dtype, act=L.act,
                     has_bias=L.b is not None, unpatchify2x2=unpatch, kernel=kernel)
    conv = x3.Conv(d, dev(L.w), None if L.b is None else dev(L.b))
    y = conv(dev(x), None if carry is None else dev(carry))
    torch.cuda.synchronize()
    return host_values(y, dtype), conv


def oracle3d(x, carry, L):
    return oracle.conv3d_causal(x.vals, L.w.vals, None if L.b is None else L.b.vals,
                                carry=None if carry is None else carry.vals, act=L.act, layout="NDHWC")


CASES_3D = [
    # (N, C_in, C_out, D, H, W, act, with_carry)
    (1, 128, 128, 2, 10, 300, "relu", True),
    (1, 128, 128, 2, 10, 300, "relu", False),
    (1, 256, 256, 1, 6, 156, "none", True),
    (2, 32, 64, 3, 7, 41, "none", True),
    (1, 40, 72, 2, 5, 19, "relu", True),      # channels not multiples of the chunk / N tile
    (1, 16, 16, 4, 1, 8, "none", True),       # a single row
    (1, 256, 128, 2, 9, 130, "none", True),
    (2, 40, 136, 3, 7, 301, "relu", True),   # two 128-channel output tiles, ragged everything
    (1, 64, 256, 2, 5, 700, "none", False),  # wide rows: several strips
]


@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", CASES_3D, ids=lambda c: "x".join(map(str, c[:6])) + ("c" if c[7] else "z"))
@pytest.mark.parametrize("kernel", ["auto", "nsub", "direct"])
def test_conv3d_causal(case, variant, kernel, monkeypatch):
    """auto: the planner's engine (the swapped 128-byte-swizzle engine when C_out >= 96);
    nsub: the positions-as-M engine forced; direct: the SIMT kernel."""
    N, Ci, Co, D, H, W, act, with_carry = case
    if kernel == "direct" and Ci * Co * H * W > 2_000_000:
        pytest.skip("the direct kernel is checked on the smaller shapes")
    if kernel == "nsub":
        monkeypatch.setenv("X3CONV_FORCE_KERNEL", "igemm_nsub")
    x, carry, L = synth.conv3d_single(C_in=Ci, C_out=Co, D=D, H=H, W=W, N=N, variant=variant, act=act,
                                      seed=3000 + sum(case[:6]), with_carry=with_carry)
    got, conv = run3d(x, carry, L, kernel="auto" if kernel == "nsub" else kernel)
    if kernel == "nsub":
        assert conv.kernel_name == "igemm_tcgen05"
    elif kernel == "auto":
        assert conv.kernel_name == ("igemm_tcgen05_sw128" if Co >= 96 else "igemm_tcgen05")
    ref = oracle3d(x, carry, L)
    if variant == "int":
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)


@pytest.mark.parametrize("shape", [(2, 9, 140), (3, 5, 300), (1, 17, 33)], ids=str)
@pytest.mark.parametrize("variant", ["sparse1", "random"])
@pytest.mark.parametrize("kernel", ["auto", "igemm"])
def test_head_clamp_unpatchify(variant, shape, kernel):
    """auto: the stencil head (one kernel, nine spatial taps in the epilogue); igemm: the single-pass
    form with kw folded into M."""
    D, H, W = shape
    x, carry, L = synth.head(D=D, H=H, W=W, variant=variant, seed=3500 + H)
    got, conv = run3d(x, carry, L, kernel=kernel, unpatch=True)
    assert conv.kernel_name == ("igemm_tcgen05_sw128_head" if kernel == "igemm" else "igemm_tcgen05_sw128_head_stencil")
    ref12 = oracle3d(x, carry, L)                                   # [1, D, H, W, 12]
    ref = oracle.unpatchify2x2(ref12.transpose(0, 4, 1, 2, 3))      # [1, 3, D, 2H, 2W]
    ref = ref.transpose(0, 2, 3, 4, 1)                              # [1, D, 2H, 2W, 3]
    assert got.shape == ref.shape
    if variant == "sparse1":
        assert_exact(got, ref, "bf16")
        assert np.max(np.abs(ref)) <= 1.0
    else:
        assert_close(got, ref)
        assert psnr(got, ref) >= PSNR_MIN
        if min(2 * H, 2 * W) >= 11:
            assert ssim_rgb(got, ref) >= SSIM_MIN


W2_CASES = [
    # (N, C_in, C_out, D, H, W, act, with_carry)
    (1, 128, 128, 2, 10, 300, "relu", True),
    (1, 128, 128, 3, 9, 140, "relu", False),
    (2, 64, 96, 2, 7, 41, "none", True),       # ragged: the pair's second window past the end
    (1, 256, 128, 2, 13, 77, "none", True),    # four channel chunks
]


@pytest.mark.parametrize("variant", ["int", "random"])
@pytest.mark.parametrize("case", W2_CASES, ids=lambda c: "x".join(map(str, c[:6])) + ("c" if c[7] else "z"))
def test_conv3d_two_window_form(case, variant, monkeypatch):
    """The two-window form (opt-in: X3CONV_W2=1; no plan takes it by default): a tile is two consecutive
    windows sharing each weight K slice."""
    monkeypatch.setenv("X3CONV_W2", "1")
    N, Ci, Co, D, H, W, act, with_carry = case
    x, carry, L = synth.conv3d_single(C_in=Ci, C_out=Co, D=D, H=H, W=W, N=N, variant=variant, act=act,
                                      seed=3300 + sum(case[:6]), with_carry=with_carry)
    got, conv = run3d(x, carry, L)
    assert x3.conv_plan_describe(conv.plan)["w2"] == 1
    ref = oracle3d(x, carry, L)
    if variant == "int":
        assert_exact(got, ref, "bf16")
    else:
        assert_close(got, ref)


# ------------------------------------------------------------------ full size, sampled (the single-pass head)

def test_full_size_head_sampled():
    x, carry, L = synth.head(seed=3950)
    got, conv = run3d(x, carry, L, kernel="igemm", unpatch=True)
    assert conv.kernel_name == "igemm_tcgen05_sw128_head"
    assert got.shape == (1, 4, 704, 1248, 3)
    seq = np.concatenate([carry.vals, x.vals], axis=1)
    pos = sample_positions(4, 352, 624, 400, seed=7)
    ref = oracle_sampled_3d(seq, L.w.vals, L.b.vals, "clamp", pos)
    g = np.stack([[got[0, t, 2 * h + (c // 2) % 2, 2 * w + c % 2, c // 4] for c in range(12)] for (t, h, w) in pos])
    assert_close(g, ref)
    assert psnr(g, ref) >= PSNR_MIN
