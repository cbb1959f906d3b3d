"""Parity at the largest sizes the boundary accepts, on sampled outputs.

conv_plan_create accepts planes of up to 2^30 positions and up to 65536 input or output channels
(larger ones are "tensor too large"); the kernels index a plane in 32 bits and tensors in 64, and the
stencil head keeps its output rows in 16 bits (more than 65535 rows go to the single-pass head). Each
case runs one layer at or next to such a limit, most with tensors far beyond 2^32 bytes, and compares
outputs with the oracle bit for bit: the whole tensor where it is small, else sampled outputs (the
corners, the first and last rows and columns, random positions; every output channel, so every
channel plane of an NCHW tensor, whose byte offsets pass 2^31 and 2^32), each from the oracle run on
that output's own zero-padded 3x3 (x 3) window.

The inputs are integer-valued, from a closed-form hash of (channel, sequence frame, row, column) that
the test evaluates with torch on the device to fill the input and again with numpy on the host for the
oracle's windows, so no oracle input comes from the device. Weights and biases are small integers
(synth's "int" and "sparse1" layers), so every fp32 partial sum is an exact integer below 2^24 and
stays inside the output type's range, and one rounding of the exact value is the only rounding: the
GPU's summation order cannot change a value (TAESD conv page, header comment and
``taesd_conv3x3_impl``: pad-1 3x3 convolution, zero outside the image; FastVideo head.cu page, header
comment: the causal 3x3x3 convolution over two carried frames and the current ones, the conv_out head
with clamp and 2x2 unpatchify).
"""
import numpy as np
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
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def hashed(c, f, h, w):
    """Input value in {-1, 0, 1} at (channel c, sequence frame f, row h, column w). Works alike on numpy
    int64 arrays and torch int64 tensors: every intermediate is non-negative and below 2^60 for
    coordinates below 2^16 (frames below 2^10)."""
    k = h * 73856093 + w * 19349663 + c * 83492791 + f * 50331653
    k = k ^ (k >> 13)
    return ((k * 40503) >> 11) % 3 - 1


def fill_nchw(x, rows=1024):
    """x [1, C, H, W] on the device <- hashed(c, 0, h, w)."""
    _, C, H, W = x.shape
    wi = torch.arange(W, device=x.device, dtype=torch.int64)[None, :]
    for c in range(C):
        for h0 in range(0, H, rows):
            hi = torch.arange(h0, min(h0 + rows, H), device=x.device, dtype=torch.int64)[:, None]
            x[0, c, h0:h0 + rows] = hashed(c, 0, hi, wi).to(x.dtype)


def fill_ndhwc(x, frame0, rows=128):
    """x [1, F, H, W, C] on the device <- hashed(c, frame0 + t, h, w)."""
    _, F, H, W, C = x.shape
    wi = torch.arange(W, device=x.device, dtype=torch.int64)[None, :, None]
    ci = torch.arange(C, device=x.device, dtype=torch.int64)[None, None, :]
    for t in range(F):
        for h0 in range(0, H, rows):
            hi = torch.arange(h0, min(h0 + rows, H), device=x.device, dtype=torch.int64)[:, None, None]
            x[0, t, h0:h0 + rows] = hashed(ci, frame0 + t, hi, wi).to(x.dtype)


def windows_2d(pos, C, H, W):
    """[P, C, 3, 3] zero-padded windows of the hashed plane around output positions (h, w)."""
    p = np.asarray(pos, np.int64)
    d = np.arange(3, dtype=np.int64) - 1
    hh = p[:, 0][:, None, None, None] + d[None, None, :, None]
    ww = p[:, 1][:, None, None, None] + d[None, None, None, :]
    cc = np.arange(C, dtype=np.int64)[None, :, None, None]
    inside = (hh >= 0) & (hh < H) & (ww >= 0) & (ww < W)
    v = hashed(cc, 0, np.clip(hh, 0, H - 1), np.clip(ww, 0, W - 1))
    return np.where(inside, v, 0).astype(np.float32)


def windows_3d(pos, C, H, W):
    """[P, 3, 3, 3, C] zero-padded windows (sequence frames t..t+2) around output positions (t, h, w)."""
    p = np.asarray(pos, np.int64)
    d = np.arange(3, dtype=np.int64)
    tt = p[:, 0][:, None, None, None, None] + d[None, :, None, None, None]
    hh = p[:, 1][:, None, None, None, None] + d[None, None, :, None, None] - 1
    ww = p[:, 2][:, None, None, None, None] + d[None, None, None, :, None] - 1
    cc = np.arange(C, dtype=np.int64)[None, None, None, None, :]
    inside = (hh >= 0) & (hh < H) & (ww >= 0) & (ww < W)
    v = hashed(cc, tt, np.clip(hh, 0, H - 1), np.clip(ww, 0, W - 1))
    return np.where(inside, v, 0).astype(np.float32)


def positions_2d(H, W, n, seed):
    rng = np.random.default_rng(seed)
    edge = (0, 1, 2, H // 2, H - 3, H - 2, H - 1)
    edge_w = (0, 1, 2, W // 2, W - 3, W - 2, W - 1)
    pos = {(h, w) for h in edge for w in edge_w if 0 <= h < H and 0 <= w < W}
    while len(pos) < n + 49:
        pos.add((int(rng.integers(H)), int(rng.integers(W))))
    return sorted(pos)


def positions_3d(D, H, W, n, seed):
    rng = np.random.default_rng(seed)
    pos = {(t, h, w) for t in range(D) for (h, w) in positions_2d(H, W, 0, seed)}
    while len(pos) < n + 49 * D:
        pos.add((int(rng.integers(D)), int(rng.integers(H)), int(rng.integers(W))))
    return sorted(pos)


def test_largest_plane_nchw_f16():
    """A 16 -> 16 NCHW f16 layer over a 32768 x 32768 plane: 2^30 positions, the largest plane the
    boundary accepts (34 GB in, 34 GB out; channel planes of 2 GB, so all but the first start past
    2^31 bytes)."""
    H = W = 32768
    C = 16
    L = synth.make_layer([9100], 2, C, C, "f16", act="relu", variant="int")
    conv = x3.Conv(x3.make_desc(2, 1, C, C, H, W, layout="NCHW", dtype="f16", act="relu"), dev(L.w), dev(L.b))
    assert conv.kernel_name == "igemm_tcgen05_sw128_nchw"
    x = torch.empty((1, C, H, W), dtype=torch.float16, device="cuda")
    fill_nchw(x)
    y = conv(x)
    del x
    pos = positions_2d(H, W, 400, seed=9101)
    hs = torch.tensor([p[0] for p in pos], device="cuda")
    ws = torch.tensor([p[1] for p in pos], device="cuda")
    got = host_values(y[0][:, hs, ws].t().contiguous(), "f16")
    del y
    ref = oracle.conv2d(windows_2d(pos, C, H, W), L.w.vals, L.b.vals, act="relu")[:, :, 1, 1]
    assert got.shape == ref.shape == (len(pos), C)
    assert_exact(got, ref, "f16")


def fill_nhwc(x, rows=64):
    """x [1, H, W, C] on the device <- hashed(c, 0, h, w)."""
    _, H, W, C = x.shape
    wi = torch.arange(W, device=x.device, dtype=torch.int64)[None, :, None]
    ci = torch.arange(C, device=x.device, dtype=torch.int64)[None, None, :]
    for h0 in range(0, H, rows):
        hi = torch.arange(h0, min(h0 + rows, H), device=x.device, dtype=torch.int64)[:, None, None]
        x[0, h0:h0 + rows] = hashed(ci, 0, hi, wi).to(x.dtype)


def test_large_plane_nhwc_taps_in_n():
    """A 64 -> 64 NHWC f16 layer over a 16384 x 16384 plane (2^28 positions, 34 GB in and 34 GB out) in
    the positions-as-M form with the horizontal taps in N and row stores by TMA, past 2^32 bytes in both
    tensors."""
    H = W = 16384
    C = 64
    L = synth.make_layer([9140], 2, C, C, "f16", act="relu", variant="int")
    conv = x3.Conv(x3.make_desc(2, 1, C, C, H, W, layout="NHWC", dtype="f16", act="relu"), dev(L.w), dev(L.b))
    g = x3.conv_plan_describe(conv.plan)
    assert conv.kernel_name == "igemm_tcgen05_sw128" and g["tn"] == 1 and g["tk"] == 0
    x = torch.empty((1, H, W, C), dtype=torch.float16, device="cuda")
    fill_nhwc(x)
    y = conv(x)
    del x
    pos = positions_2d(H, W, 400, seed=9141)
    hs = torch.tensor([p[0] for p in pos], device="cuda")
    ws = torch.tensor([p[1] for p in pos], device="cuda")
    got = host_values(y[0][hs, ws].contiguous(), "f16")
    del y
    ref = oracle.conv2d(windows_2d(pos, C, H, W), L.w.vals, L.b.vals, act="relu")[:, :, 1, 1]
    assert got.shape == ref.shape == (len(pos), C)
    assert_exact(got, ref, "f16")


@pytest.mark.parametrize("C_in,C_out", [(65536, 16), (16, 65536)], ids=["cin65536", "cout65536"])
def test_most_channels_nchw_f16(C_in, C_out):
    """The most input channels (1024 staged 64-channel chunks per tile) and the most output channels
    (512 channel tiles) the boundary accepts, 8 x 8 plane, every output compared."""
    H = W = 8
    L = synth.make_layer([9110, C_in, C_out], 2, C_in, C_out, "f16", variant="int")
    conv = x3.Conv(x3.make_desc(2, 1, C_in, C_out, H, W, layout="NCHW", dtype="f16"), dev(L.w), dev(L.b))
    hi = np.arange(H, dtype=np.int64)[None, :, None]
    wi = np.arange(W, dtype=np.int64)[None, None, :]
    ci = np.arange(C_in, dtype=np.int64)[:, None, None]
    xv = hashed(ci, 0, hi, wi).astype(np.float32)[None]
    x = torch.from_numpy(xv).to(torch.float16).cuda()
    got = host_values(conv(x), "f16")
    ref = oracle.conv2d(xv, L.w.vals, L.b.vals)
    # premise of exactness: no partial sum reaches 2^24, and no output leaves f16's range
    assert np.max(np.abs(ref)) < 60000.0
    assert got.shape == ref.shape
    assert_exact(got, ref, "f16")


def test_causal_layer_past_4gb():
    """A causal 128 -> 128 bf16 NDHWC layer over 8 frames (+2 carried) at 2048 x 2048: input, carry and
    output 8.6, 2.1 and 8.6 GB, so frame offsets pass 2^32 bytes; sampled outputs of every frame,
    the first two reading the carried frames."""
    D, H, W, C = 8, 2048, 2048, 128
    L = synth.make_layer([9120], 3, C, C, "bf16", act="relu", variant="int")
    conv = x3.Conv(x3.make_desc(3, 1, C, C, H, W, D=D, layout="NDHWC", dtype="bf16", act="relu"),
                   dev(L.w), dev(L.b))
    assert conv.kernel_name == "igemm_tcgen05_sw128"
    x = torch.empty((1, D, H, W, C), dtype=torch.bfloat16, device="cuda")
    carry = torch.empty((1, 2, H, W, C), dtype=torch.bfloat16, device="cuda")
    fill_ndhwc(carry, 0)
    fill_ndhwc(x, 2)
    y = conv(x, carry)
    del x, carry
    pos = positions_3d(D, H, W, 300, seed=9121)
    idx = [torch.tensor([p[i] for p in pos], device="cuda") for i in range(3)]
    got = host_values(y[0][idx[0], idx[1], idx[2]].contiguous(), "bf16")
    del y
    cr = windows_3d(pos, C, H, W)
    ref = oracle.conv3d_causal(cr[:, 2:3], L.w.vals, L.b.vals, carry=cr[:, 0:2], act="relu",
                               layout="NDHWC")[:, 0, 1, 1, :]
    assert got.shape == ref.shape == (len(pos), C)
    assert_exact(got, ref, "bf16")


@pytest.mark.parametrize("H,kernel", [(65535, "igemm_tcgen05_sw128_head_stencil"),
                                      (65536, "igemm_tcgen05_sw128_head")], ids=["stencil65535", "single65536"])
def test_head_most_rows(H, kernel):
    """The conv_out head (256 -> 12, clamp, 2x2 unpatchify) over 3 frames (+2 carried) of H x 64: the
    stencil head at its largest height (65535 output rows, its run table's 16-bit rows), and one row
    more, which the planner gives to the single-pass head; sampled 2 x 2 RGB blocks of every frame."""
    D, W, C = 3, 64, 256
    L = synth.make_layer([9130], 3, C, 12, "bf16", act="clamp", variant="sparse1")
    conv = x3.Conv(x3.make_desc(3, 1, C, 12, H, W, D=D, layout="NDHWC", dtype="bf16", act="clamp",
                                unpatchify2x2=True), dev(L.w), dev(L.b))
    assert conv.kernel_name == kernel
    x = torch.empty((1, D, H, W, C), dtype=torch.bfloat16, device="cuda")
    carry = torch.empty((1, 2, H, W, C), dtype=torch.bfloat16, device="cuda")
    fill_ndhwc(carry, 0, rows=1024)
    fill_ndhwc(x, 2, rows=1024)
    y = conv(x, carry)
    del x, carry
    assert tuple(y.shape) == (1, D, 2 * H, 2 * W, 3)
    pos = positions_3d(D, H, W, 300, seed=9131 + H)
    t, h, w = (torch.tensor([p[i] for p in pos], device="cuda") for i in range(3))
    dy = torch.arange(2, device="cuda")
    blk = y[0][t[:, None, None], 2 * h[:, None, None] + dy[None, :, None], 2 * w[:, None, None] + dy[None, None, :]]
    got = host_values(blk.contiguous(), "bf16")                      # [P, 2, 2, 3]
    del y
    cr = windows_3d(pos, C, H, W)
    y12 = oracle.conv3d_causal(cr[:, 2:3], L.w.vals, L.b.vals, carry=cr[:, 0:2], act="clamp",
                               layout="NDHWC")[:, 0, 1, 1, :]          # [P, 12]
    rgb = oracle.unpatchify2x2(y12[:, :, None, None, None])[:, :, 0]  # [P, 3, 2, 2]
    ref = rgb.transpose(0, 2, 3, 1)
    assert got.shape == ref.shape == (len(pos), 2, 2, 3)
    assert_exact(got, ref, "bf16")
    assert 0.0 < np.mean(np.abs(ref) < 1.0)  # unclamped values are present
