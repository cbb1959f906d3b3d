"""Seeded sweeps through the C ABI against the oracle: random layer shapes, random 2D and causal stacks,
random layers cut into random row bands, and random conv_out head planes.

Each case draws its descriptor from a fixed generator: 2D layers (NCHW or NHWC, f16 or bf16, stride 1
or 2) or causal 3D layers (NDHWC bf16, with or without a history), channel counts around and between
the engines' tile sizes, heights and widths from one row or column to a few tiles with ragged tails,
batches of 1 to 3 and every activation (TAESD conv page: pad-1 cross-correlation with stride, bias,
ReLU; FastVideo head.cu page, header comment: causal 3x3x3 over [2 carried frames, current frames],
all taps in one fp32 accumulator, clamp). Data are integers in {-2..2}, so every fp32 partial sum is an
exact integer below 2^24 and the stored values must equal the oracle's, rounded once to the storage
type, bit for bit, whatever engine or form the planner picks for the shape. The sweep must reach the
tensor-core engines and the direct kernel.
"""
import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_exact, dev, host_values

pytestmark = pytest.mark.gpu

N_2D, N_3D = 28, 20
MAX_FLOP = 1.5e10  # keeps the oracle at a few seconds per case


def _draw(seed=7100):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < N_2D:
        c = dict(dims=2, layout=str(rng.choice(["NCHW", "NHWC"])), dtype=str(rng.choice(["f16", "bf16"])),
                 C_in=int(rng.choice([1, 3, 8, 16, 24, 40, 64, 72, 128])),
                 C_out=int(rng.choice([8, 16, 32, 48, 64, 80, 96, 128, 136])),
                 stride=int(rng.choice([1, 1, 2])), N=int(rng.integers(1, 4)), H=int(rng.integers(1, 70)),
                 W=int(rng.integers(1, 150)), act=str(rng.choice(["none", "relu", "clamp"])))
        if 2.0 * 9 * c["C_in"] * c["C_out"] * c["N"] * c["H"] * c["W"] <= MAX_FLOP:
            cases.append(c)
    while len(cases) < N_2D + N_3D:
        c = dict(dims=3, layout="NDHWC", dtype="bf16", C_in=int(rng.choice([8, 16, 32, 40, 64, 128, 256])),
                 C_out=int(rng.choice([8, 16, 64, 72, 96, 128, 256])), stride=1, N=int(rng.integers(1, 3)),
                 D=int(rng.integers(1, 5)), H=int(rng.integers(1, 21)), W=int(rng.integers(1, 200)),
                 act=str(rng.choice(["none", "relu", "clamp"])), carry=bool(rng.integers(0, 2)))
        if 2.0 * 27 * c["C_in"] * c["C_out"] * c["N"] * c["D"] * c["H"] * c["W"] <= MAX_FLOP:
            cases.append(c)
    return cases


CASES = _draw()
SEEN = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def _run(i, c):
    seed = [7200, i]
    if c["dims"] == 2:
        shape = (c["N"], c["C_in"], c["H"], c["W"]) if c["layout"] == "NCHW" else (c["N"], c["H"], c["W"], c["C_in"])
        x = synth.activation(seed + [0], shape, c["dtype"], "int")
        L = synth.make_layer(seed, 2, c["C_in"], c["C_out"], c["dtype"], stride=c["stride"], act=c["act"], variant="int")
        d = x3.make_desc(2, c["N"], c["C_in"], c["C_out"], c["H"], c["W"], stride=c["stride"], layout=c["layout"],
                         dtype=c["dtype"], act=c["act"])
        conv = x3.Conv(d, dev(L.w), dev(L.b))
        got = host_values(conv(dev(x)), c["dtype"])
        ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, stride=c["stride"], act=c["act"], layout=c["layout"])
    else:
        x = synth.activation(seed + [0], (c["N"], c["D"], c["H"], c["W"], c["C_in"]), "bf16", "int")
        carry = synth.activation(seed + [1], (c["N"], 2, c["H"], c["W"], c["C_in"]), "bf16", "int") if c["carry"] else None
        L = synth.make_layer(seed, 3, c["C_in"], c["C_out"], "bf16", act=c["act"], variant="int")
        d = x3.make_desc(3, c["N"], c["C_in"], c["C_out"], c["H"], c["W"], D=c["D"], layout="NDHWC", dtype="bf16",
                         act=c["act"])
        conv = x3.Conv(d, dev(L.w), dev(L.b))
        got = host_values(conv(dev(x), None if carry is None else dev(carry)), "bf16")
        ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=None if carry is None else carry.vals,
                                   act=c["act"], layout="NDHWC")
    torch.cuda.synchronize()
    return got, ref, conv.kernel_name


@pytest.mark.parametrize("i", range(len(CASES)))
def test_random_shape_matches_oracle(i):
    c = CASES[i]
    got, ref, kname = _run(i, c)
    SEEN[i] = kname
    assert got.shape == ref.shape, (c, got.shape, ref.shape)
    assert_exact(got, ref, c["dtype"])


def test_sweep_reaches_every_engine():
    """Runs after the cases (pytest keeps file order): the planner sent the sweep's shapes to the
    swapped-operand tensor-core engine, to another tensor-core form or engine, and to the direct kernel."""
    if len(SEEN) < len(CASES):
        for i in range(len(CASES)):
            if i not in SEEN:
                SEEN[i] = _run(i, CASES[i])[2]
    names = set(SEEN.values())
    assert any(n.startswith("igemm_tcgen05_sw128") for n in names), names
    assert any(n.startswith("igemm_tcgen05") for n in names), names
    assert "direct_simt" in names, names


def _draw_stacks(n=10, seed=7300):
    """2D NCHW stacks of 2 to 5 layers: channel counts that are multiples of 8 after the first layer
    (the channels-last stack path), stride 2 anywhere but the last layer."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        depth = int(rng.integers(2, 6))
        chans = [int(rng.choice([1, 3, 8, 16]))] + [int(rng.choice([8, 16, 32, 48, 64, 72])) for _ in range(depth)]
        strides = [int(rng.choice([1, 1, 2])) for _ in range(depth - 1)] + [1]
        out.append(dict(N=int(rng.integers(1, 3)), H=int(rng.integers(8, 60)), W=int(rng.integers(8, 130)),
                        dtype=str(rng.choice(["f16", "bf16"])), chans=chans, strides=strides))
    return out


STACKS = _draw_stacks()


@pytest.mark.parametrize("i", range(len(STACKS)))
def test_random_stack_matches_oracle(i):
    """'fewtaps' data (integer inputs, three +-1 weights per output channel, integer bias) keep every
    value of the chain an exact integer, so the stack's output equals the oracle's chain with the
    intermediates rounded to the storage type bit for bit."""
    c = STACKS[i]
    x = synth.activation([7400, i, 0], (c["N"], c["chans"][0], c["H"], c["W"]), c["dtype"], "fewtaps")
    layers = [synth.make_layer([7400, i, 1 + k], 2, ci, co, c["dtype"], stride=s, act="relu", variant="fewtaps")
              for k, (ci, co, s) in enumerate(zip(c["chans"][:-1], c["chans"][1:], c["strides"]))]
    convs, h, w = [], c["H"], c["W"]
    for L in layers:
        convs.append(x3.Conv(x3.make_desc(2, c["N"], L.C_in, L.C_out, h, w, stride=L.stride, dtype=c["dtype"],
                                          act="relu"), dev(L.w), dev(L.b)))
        h, w = convs[-1].H_out, convs[-1].W_out
    got = host_values(x3.ConvStack(convs)(dev(x)), c["dtype"])
    torch.cuda.synchronize()
    y = x.vals
    for L in layers:
        y, _ = oracle.round_to(oracle.conv2d(y, L.w.vals, L.b.vals, stride=L.stride, act="relu"), c["dtype"])
    assert got.shape == y.shape
    assert np.array_equal(got, y)


def _draw_stacks3d(n=6, seed=7500):
    """Causal 3D stacks of 2 or 3 layers (channels-last bf16) run as two passes with their histories."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        depth = int(rng.integers(2, 4))
        chans = [int(rng.choice([8, 16, 32, 64]))] + [int(rng.choice([16, 32, 64, 96, 128])) for _ in range(depth)]
        out.append(dict(N=int(rng.integers(1, 3)), D=int(rng.integers(1, 5)), H=int(rng.integers(1, 13)),
                        W=int(rng.integers(8, 150)), chans=chans,
                        acts=[str(rng.choice(["relu", "none"])) for _ in range(depth)]))
    return out


STACKS3D = _draw_stacks3d()


def _oracle_pass(x, carries, layers):
    """Layer by layer, each output rounded to bf16 as the library stores it; the new histories are the
    last two frames of each layer's input sequence [history, input]."""
    y, new = x, []
    for i, L in enumerate(layers):
        seq = np.concatenate([carries[i], y], axis=1)
        new.append(seq[:, -2:].copy())
        y, _ = oracle.round_to(oracle.conv3d_causal(y, L.w.vals, L.b.vals, carry=carries[i], act=L.act,
                                                    layout="NDHWC"), "bf16")
    return y, new


@pytest.mark.parametrize("i", range(len(STACKS3D)))
def test_random_causal_stack_two_passes(i):
    """Two passes of a random causal stack: the first with no history (zeros), the second reading the
    histories the first wrote; outputs and the final histories bit for bit against the oracle on
    'fewtaps' data (integer inputs, three +-1 weights per output channel: exact integer chains)."""
    c = STACKS3D[i]
    N, D, H, W, chans = c["N"], c["D"], c["H"], c["W"], c["chans"]
    layers = [synth.make_layer([7600, i, k], 3, ci, co, "bf16", act=a, variant="fewtaps")
              for k, (ci, co, a) in enumerate(zip(chans[:-1], chans[1:], c["acts"]))]
    convs = [x3.Conv(x3.make_desc(3, N, L.C_in, L.C_out, H, W, D=D, act=L.act), dev(L.w), dev(L.b)) for L in layers]
    stack = x3.ConvStack(convs)
    cdev = [torch.zeros((N, 2, H, W, ci), dtype=torch.bfloat16, device="cuda") for ci in chans[:-1]]
    chost = [np.zeros((N, 2, H, W, ci), np.float32) for ci in chans[:-1]]
    for p in range(2):
        x = synth.activation([7600, i, 10 + p], (N, D, H, W, chans[0]), "bf16", "fewtaps")
        got = host_values(stack(dev(x), carries=cdev, carry_valid=p > 0), "bf16")
        torch.cuda.synchronize()
        want, chost = _oracle_pass(x.vals, chost, layers)
        assert got.shape == want.shape
        assert np.array_equal(got, want), (c, p)
        for k in range(len(layers)):
            assert np.array_equal(host_values(cdev[k], "bf16"), chost[k]), (c, p, k)


def _draw_bands(n=8, seed=7700):
    """Random stride-1 layers (2D NHWC, 2D NCHW, causal 3D) cut into 2 to 4 random row bands."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        dims = int(rng.choice([2, 2, 3]))
        H = int(rng.integers(4, 60))
        cuts = sorted(set(int(v) for v in rng.integers(1, H, size=int(rng.integers(1, 4)))))
        bounds = [0] + cuts + [H]
        c = dict(dims=dims, N=int(rng.integers(1, 3)), H=H, W=int(rng.integers(8, 140)),
                 C_in=int(rng.choice([8, 16, 64, 128])), C_out=int(rng.choice([16, 64, 96, 128])),
                 act=str(rng.choice(["none", "relu"])), bands=[(a, b - a) for a, b in zip(bounds[:-1], bounds[1:])])
        if dims == 2:
            c.update(layout=str(rng.choice(["NHWC", "NCHW"])), dtype=str(rng.choice(["f16", "bf16"])))
            if c["layout"] == "NCHW":
                c["W"] = (c["W"] + 7) // 8 * 8  # the NCHW tensor-core form stages 16-byte rows
        else:
            c.update(layout="NDHWC", dtype="bf16", D=int(rng.integers(1, 4)))
        out.append(c)
    return out


BANDS = _draw_bands()


@pytest.mark.parametrize("i", range(len(BANDS)))
def test_random_bands_concatenate_to_the_plane(i):
    """Banded mode (FastVideo head.cu page: head_stencil_kernel's band row offset and global height):
    each band computed from its rows plus the halo rows that exist; the bands, concatenated, equal the
    whole plane bit for bit, and the plane equals the oracle on integer data."""
    c = BANDS[i]
    dt, H, W, N = c["dtype"], c["H"], c["W"], c["N"]
    if c["dims"] == 3:
        x = synth.activation([7800, i, 0], (N, c["D"], H, W, c["C_in"]), dt, "int")
        carry = synth.activation([7800, i, 1], (N, 2, H, W, c["C_in"]), dt, "int")
        L = synth.make_layer([7800, i], 3, c["C_in"], c["C_out"], dt, act=c["act"], variant="int")
        base = dict(dims=3, N=N, C_in=c["C_in"], C_out=c["C_out"], D=c["D"], W=W, layout="NDHWC", dtype=dt, act=c["act"])
        ax = 2
    else:
        shape = (N, c["C_in"], H, W) if c["layout"] == "NCHW" else (N, H, W, c["C_in"])
        x = synth.activation([7800, i, 0], shape, dt, "int")
        carry = None
        L = synth.make_layer([7800, i], 2, c["C_in"], c["C_out"], dt, act=c["act"], variant="int")
        base = dict(dims=2, N=N, C_in=c["C_in"], C_out=c["C_out"], W=W, layout=c["layout"], dtype=dt, act=c["act"])
        ax = 2 if c["layout"] == "NCHW" else 1
    full = x3.Conv(x3.make_desc(H=H, **base), dev(L.w), dev(L.b))
    xd, cd = dev(x), (dev(carry) if carry is not None else None)
    y_full = full(xd, cd) if cd is not None else full(xd)
    outs = []
    for lo, rows in c["bands"]:
        in_lo, in_hi = x3.band_input_rows(lo, rows, H)
        conv = x3.Conv(x3.make_desc(H=in_hi - in_lo, band_lo=lo, band_rows=rows, H_global=H, **base), dev(L.w), dev(L.b))
        assert conv.kernel_name == full.kernel_name
        xb = xd.narrow(ax, in_lo, in_hi - in_lo).contiguous()
        if cd is not None:
            outs.append(conv(xb, cd.narrow(ax, in_lo, in_hi - in_lo).contiguous()))
        else:
            outs.append(conv(xb))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, dim=ax), y_full), c
    got = host_values(y_full, dt)
    if c["dims"] == 3:
        ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act=c["act"], layout="NDHWC")
    else:
        ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, act=c["act"], layout=c["layout"])
    assert_exact(got, ref, dt)


def _draw_heads(n=8, seed=7900):
    rng = np.random.default_rng(seed)
    return [dict(N=int(rng.integers(1, 3)), D=int(rng.integers(1, 5)), H=int(rng.integers(1, 60)),
                 W=int(rng.integers(1, 120)), carry=bool(rng.integers(0, 2))) for _ in range(n)]


HEADS = _draw_heads()


@pytest.mark.parametrize("i", range(len(HEADS)))
def test_random_head_shapes(i):
    """The conv_out head (256 -> 12, clamp, 2x2 unpatchify; the stencil head, the default) on random
    plane sizes, with and without history: exact on sparse {-1,0,1} weights (small sums, mostly
    unclamped), and on random data bit for bit the split head with fp32 G (same fp32 sums, same order)."""
    c = HEADS[i]
    N, D, H, W = c["N"], c["D"], c["H"], c["W"]
    for variant in ("sparse1", "random"):
        x = synth.activation([8000, i, 0], (N, D, H, W, 256), "bf16", variant, ("normal", 1.0))
        carry = synth.activation([8000, i, 1], (N, 2, H, W, 256), "bf16", variant, ("normal", 1.0)) if c["carry"] else None
        L = synth.make_layer([8000, i], 3, 256, 12, "bf16", act="clamp", variant=variant, bias_range=0.05)
        outs = {}
        for kernel in ("auto", "head_split"):
            d = x3.make_desc(3, N, 256, 12, H, W, D=D, layout="NDHWC", dtype="bf16", act="clamp", unpatchify2x2=True,
                             kernel=kernel)
            conv = x3.Conv(d, dev(L.w), dev(L.b))
            if kernel == "auto":
                assert conv.kernel_name == "igemm_tcgen05_sw128_head_stencil"
            outs[kernel] = host_values(conv(dev(x), None if carry is None else dev(carry)), "bf16")
        torch.cuda.synchronize()
        y12 = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=None if carry is None else carry.vals,
                                   act="clamp", layout="NDHWC")
        ref = oracle.unpatchify2x2(y12.transpose(0, 4, 1, 2, 3)).transpose(0, 2, 3, 4, 1)
        assert outs["auto"].shape == ref.shape == (N, D, 2 * H, 2 * W, 3)
        if variant == "sparse1":
            assert_exact(outs["auto"], ref, "bf16")
        assert np.array_equal(outs["auto"], outs["head_split"])
