"""GPU parity of the banded (row-band) mode: the layer computes output rows [band_lo, band_lo + rows) of
an H_global-row image from an input holding the band's rows plus the halo rows that exist globally
(FastVideo head.cu page, head_stencil_kernel and its wrapper: band offset, global height, rows outside
the plane skipped). Bands of one plane, concatenated, must equal the whole plane's output bit for bit,
and on integer data the whole plane equals the oracle. Each engine and form is covered: the channels-
last tensor-core engine (128-row, positions-as-M, M = 64, NCHW, stencil head, single-pass head), the
positions-as-M engine of 3D layers with fewer than 96 output channels, and the direct kernel."""
import pytest
import torch

import bench
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
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


FORMS = {
    # name: (descriptor of the whole plane, environment, expected kernel name prefix)
    "causal128_cl": (dict(dims=3, N=1, C_in=128, C_out=128, D=2, H=37, W=70, act="relu"), {}, "igemm_tcgen05_sw128"),
    "causal64_igemm": (dict(dims=3, N=1, C_in=64, C_out=64, D=2, H=21, W=45), {}, "igemm_tcgen05"),
    "nhwc64_tn": (dict(dims=2, N=2, C_in=64, C_out=64, H=29, W=61, layout="NHWC", dtype="f16", act="relu"), {},
                  "igemm_tcgen05_sw128"),
    "nhwc64_m64": (dict(dims=2, N=2, C_in=64, C_out=64, H=29, W=61, layout="NHWC", dtype="f16", act="relu"),
                   {"X3CONV_TN": "0"}, "igemm_tcgen05_sw128"),
    "nchw16": (dict(dims=2, N=1, C_in=16, C_out=16, H=33, W=64, layout="NCHW", dtype="f16", act="relu"), {},
               "igemm_tcgen05_sw128_nchw"),
    "direct": (dict(dims=3, N=1, C_in=8, C_out=8, D=2, H=11, W=13, kernel="direct"), {}, "direct_simt"),
    "head_stencil": (dict(dims=3, N=1, C_in=256, C_out=12, D=2, H=30, W=40, act="clamp", unpatchify2x2=True), {},
                     "igemm_tcgen05_sw128_head_stencil"),
    # large enough that every band's CTAs run several abutting windows (row sums carried across seams)
    "head_stencil_runs": (dict(dims=3, N=1, C_in=256, C_out=12, D=2, H=180, W=560, act="clamp", unpatchify2x2=True),
                          {}, "igemm_tcgen05_sw128_head_stencil"),
    "head_single_pass": (dict(dims=3, N=1, C_in=256, C_out=12, D=2, H=30, W=40, act="clamp", unpatchify2x2=True,
                              kernel="igemm"), {}, "igemm_tcgen05_sw128_head"),
}


def row_axis(d):
    lay = d.get("layout", "NDHWC" if d["dims"] == 3 else "NCHW")
    return {"NCHW": 2, "NHWC": 1, "NCDHW": 3, "NDHWC": 2}[lay]


def bands_of(H):
    a, b = max(1, H // 3), max(2, (2 * H) // 3 + 1)
    return [(0, a), (a, b - a), (b, H - b)]


def run_bands(d, L, x, carry, bands):
    """The whole plane and each band (input rows sliced with their halo), on the GPU."""
    ax = row_axis(d)
    H = d["H"]
    full = x3.Conv(x3.make_desc(**d), dev(L.w), dev(L.b))
    xd, cd = dev(x), (dev(carry) if carry is not None else None)
    y_full = full(xd, cd)
    outs = []
    for lo, rows in bands:
        in_lo, in_hi = x3.band_input_rows(lo, rows, H)
        db = dict(d, H=in_hi - in_lo, band_lo=lo, band_rows=rows, H_global=H)
        conv = x3.Conv(x3.make_desc(**db), dev(L.w), dev(L.b))
        assert conv.kernel_name == full.kernel_name
        xb = xd.narrow(ax, in_lo, in_hi - in_lo).contiguous()
        cb = cd.narrow(ax, in_lo, in_hi - in_lo).contiguous() if cd is not None else None
        outs.append(conv(xb, cb))
    torch.cuda.synchronize()
    return full, y_full, outs


@pytest.mark.parametrize("name", sorted(FORMS))
def test_bands_concatenate_to_the_plane(name, monkeypatch):
    d, env, kname = FORMS[name]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    dtype = d.get("dtype", "bf16")
    key = 6100 + len(name)
    if d["dims"] == 3:
        shape = (d["N"], d["D"], d["H"], d["W"], d["C_in"])
        x = synth.activation([key, 0], shape, dtype, "int")
        carry = synth.activation([key, 3], (d["N"], 2, d["H"], d["W"], d["C_in"]), dtype, "int")
        variant = "sparse1" if d.get("unpatchify2x2") else "int"
        L = synth.make_layer([key], 3, d["C_in"], d["C_out"], dtype, act=d.get("act", "none"), variant=variant)
    else:
        lay = d["layout"]
        shape = (d["N"], d["C_in"], d["H"], d["W"]) if lay == "NCHW" else (d["N"], d["H"], d["W"], d["C_in"])
        x = synth.activation([key, 0], shape, dtype, "int")
        carry = None
        L = synth.make_layer([key], 2, d["C_in"], d["C_out"], dtype, act=d.get("act", "none"), variant="int")
    full, y_full, outs = run_bands(d, L, x, carry, bands_of(d["H"]))
    assert full.kernel_name.startswith(kname), full.kernel_name
    oax = row_axis(d)
    assert torch.equal(torch.cat(outs, dim=oax), y_full)
    # the whole plane against the oracle (integer / sparse data: exact)
    got = host_values(y_full, dtype)
    if d["dims"] == 3:
        ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act=d.get("act", "none"),
                                   layout="NDHWC")
        if d.get("unpatchify2x2"):
            ref = oracle.unpatchify2x2(ref.transpose(0, 4, 1, 2, 3)).transpose(0, 2, 3, 4, 1)
    else:
        ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, act=d.get("act", "none"), layout=d["layout"])
    assert_exact(got, ref, dtype)


def test_bands_of_the_full_size_causal_layer():
    """The causal 128->128 layer at 4+2 x 352x624 (the benchmark's plan) in three bands on integer
    data: the bands concatenate to the whole plane bit for bit, which equals the oracle."""
    d = dict(bench.layer_descs()["stack"][0])
    x, carry, L = synth.conv3d_single(C_in=128, C_out=128, D=4, H=352, W=624, variant="int", act="relu", seed=6201)
    full, y_full, outs = run_bands(d, L, x, carry, [(0, 100), (100, 137), (237, 115)])
    assert torch.equal(torch.cat(outs, dim=2), y_full)
    ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="relu", layout="NDHWC")
    assert_exact(host_values(y_full, "bf16"), ref, "bf16")
