"""Pins of the CPU oracle to things other than itself (CPU only).

Each check would fail under a plausible mistake in the oracle: a flipped kernel (convolution
instead of cross-correlation), a wrong padding offset, a transposed weight, a wrong stride
mapping, a wrong temporal order, a dropped bias or a misplaced activation. ``test_oracle_mutants``
plants such mistakes in a copy of the oracle and checks that these pins catch them.

Definitions: musetalk-bench patches/taesd_conv.cuh.new (taesd_conv3x3_impl) for the 2D
operation; FastVideo wan22_vae_decode/solution/head.cu (header comment, head_stencil_kernel) for
the causal 3x3x3 head with bias, clamp and fp32 accumulation of all 27 taps.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
U = 2.0 ** -24


def brute_conv2d_f64(x, w, b, stride, act):
    """float64 brute force: every output a dot product over (ci,kh,kw) with zero padding."""
    N, C, H, W = x.shape
    Co = w.shape[0]
    Ho, Wo = (H - 1) // stride + 1, (W - 1) // stride + 1
    xp = np.zeros((N, C, H + 2, W + 2))
    xp[:, :, 1:H + 1, 1:W + 1] = x
    y = np.zeros((N, Co, Ho, Wo))
    absy = np.zeros_like(y)
    for oh in range(Ho):
        for ow in range(Wo):
            win = xp[:, :, stride * oh:stride * oh + 3, stride * ow:stride * ow + 3]
            y[:, :, oh, ow] = np.einsum("ncij,ocij->no", win, w)
            absy[:, :, oh, ow] = np.einsum("ncij,ocij->no", np.abs(win), np.abs(w))
    if b is not None:
        y += b[None, :, None, None]
        absy += np.abs(b)[None, :, None, None]
    return _act(y, act), absy


def brute_conv3d_f64(x, w, b, carry, act):
    N, C, D, H, W = x.shape
    Co = w.shape[0]
    c = np.zeros((N, C, 2, H, W)) if carry is None else carry
    xt = np.concatenate([c, x], axis=2)
    xp = np.zeros((N, C, D + 2, H + 2, W + 2))
    xp[:, :, :, 1:H + 1, 1:W + 1] = xt
    y = np.zeros((N, Co, D, H, W))
    absy = np.zeros_like(y)
    for t in range(D):
        for h in range(H):
            for ww in range(W):
                win = xp[:, :, t:t + 3, h:h + 3, ww:ww + 3]
                y[:, :, t, h, ww] = np.einsum("ncijk,ocijk->no", win, w)
                absy[:, :, t, h, ww] = np.einsum("ncijk,ocijk->no", np.abs(win), np.abs(w))
    if b is not None:
        y += b[None, :, None, None, None]
        absy += np.abs(b)[None, :, None, None, None]
    return _act(y, act), absy


def _act(y, act):
    if act == "relu":
        return np.maximum(y, 0)
    if act == "clamp":
        return np.clip(y, -1, 1)
    return y


def within_fp32_sum_bound(got, ref, absref, nterms):
    gamma = nterms * U / (1 - nterms * U)
    return np.all(np.abs(got.astype(np.float64) - ref) <= gamma * absref + 1e-30)


# ------------------------------------------------------------------ rounding (IEEE 754 RNE)

def test_f16_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle_mod.decode_bits(bits, "f16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _tie_heavy_f32(rng, n):
    """Random f32 values plus exact midpoints between neighbouring f16 and bf16 values."""
    r = rng.standard_normal(n).astype(np.float32) * np.float32(4.0) ** rng.integers(-12, 9, n)
    h = rng.integers(0, 0x7bff, n).astype(np.uint16).view(np.float16).astype(np.float64)
    h2 = (rng.integers(0, 0x7bff, n).astype(np.uint16) + 1).view(np.float16).astype(np.float64)
    mids16 = ((h + h2) / 2).astype(np.float32)
    bf = rng.integers(0, 0x7f7f, n).astype(np.uint32) << 16
    mids_bf = (bf | 0x8000).view(np.float32)
    edge = np.array([65504, 65519.99, 65520, 65536, 1e-8, 2 ** -25, 2 ** -24, 3 * 2 ** -26,
                     6.0e-5, 6.1035156e-05, -0.0, 0.0, np.inf, -np.inf], np.float32)
    return np.concatenate([r, mids16, -mids16, mids_bf, -mids_bf, edge])


def test_f16_encode_matches_numpy(oracle_mod):
    x = _tie_heavy_f32(np.random.default_rng(5), 20000)
    _, bits = oracle_mod.round_to(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(bits, ref)


def test_bf16_encode_matches_torch(oracle_mod):
    x = _tie_heavy_f32(np.random.default_rng(6), 20000)
    _, bits = oracle_mod.round_to(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)


# ------------------------------------------------------------------ hand-worked values

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_values(oracle_mod, case):
    if case["kind"] == "conv2d":
        x = np.array(case["x"], np.float32)[None, None]
        w = np.array(case["w"], np.float32)[None, None]
        y = oracle_mod.conv2d(x, w, np.array(case["bias"], np.float32), stride=case["stride"],
                              act=case["act"])
        assert np.array_equal(y[0, 0], np.array(case["y"], np.float32))
    else:
        x = np.array(case["x"], np.float32).reshape(1, 1, -1, 1, 1)
        w = np.zeros((1, 1, 3, 3, 3), np.float32)
        w[0, 0, :, 1, 1] = case["wt"]
        carry = None if case["carry"] is None else np.array(case["carry"], np.float32).reshape(1, 1, 2, 1, 1)
        y = oracle_mod.conv3d_causal(x, w, np.array(case["bias"], np.float32), carry=carry,
                                     act=case["act"])
        assert np.array_equal(y.ravel(), np.array(case["y"], np.float32))


# ------------------------------------------------------------------ brute force + library

SHAPES_2D = [(1, 1, 1, 1, 1), (1, 2, 3, 2, 3), (2, 3, 5, 5, 7), (1, 5, 2, 7, 5), (1, 3, 4, 1, 6)]


@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("shape", SHAPES_2D)
def test_conv2d_vs_brute_force(oracle_mod, shape, stride):
    N, Ci, Co, H, W = shape
    rng = np.random.default_rng(hash((shape, stride)) & 0xffff)
    x = rng.uniform(-1, 1, (N, Ci, H, W)).astype(np.float32)
    w = rng.normal(0, 0.3, (Co, Ci, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    for act in ("none", "relu"):
        y = oracle_mod.conv2d(x, w, b, stride=stride, act=act)
        ref, absref = brute_conv2d_f64(x.astype(np.float64), w.astype(np.float64),
                                       b.astype(np.float64), stride, act)
        assert y.shape == ref.shape
        assert within_fp32_sum_bound(y, ref, absref, 9 * Ci + 1)


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 1), (1, 2, 3, 2, 3, 4), (2, 3, 2, 3, 4, 2),
                                   (1, 5, 1, 1, 2, 5)])
@pytest.mark.parametrize("with_carry", [False, True])
def test_conv3d_vs_brute_force(oracle_mod, shape, with_carry):
    N, Ci, Co, D, H, W = shape
    rng = np.random.default_rng(7 + sum(shape))
    x = rng.normal(0, 1, (N, Ci, D, H, W)).astype(np.float32)
    c = rng.normal(0, 1, (N, Ci, 2, H, W)).astype(np.float32) if with_carry else None
    w = rng.normal(0, 0.2, (Co, Ci, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    for act in ("none", "relu", "clamp"):
        y = oracle_mod.conv3d_causal(x, w, b, carry=c, act=act)
        ref, absref = brute_conv3d_f64(x.astype(np.float64), w.astype(np.float64),
                                       b.astype(np.float64),
                                       None if c is None else c.astype(np.float64), act)
        assert within_fp32_sum_bound(y, ref, absref, 27 * Ci + 1)


@pytest.mark.parametrize("variant", ["int", "random"])
def test_conv2d_integer_exact_vs_int64(oracle_mod, variant):
    """On {-2..2} integers every fp32 partial sum is exact, so the oracle equals int64 math."""
    rng = np.random.default_rng(11)
    x = rng.integers(-2, 3, (2, 6, 9, 11))
    w = rng.integers(-2, 3, (5, 6, 3, 3))
    b = rng.integers(-2, 3, 5)
    for stride in (1, 2):
        y = oracle_mod.conv2d(x, w, b, stride=stride, act="relu")
        ref, _ = brute_conv2d_f64(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64),
                                  stride, "relu")
        assert np.array_equal(y.astype(np.int64), ref.astype(np.int64))
        assert np.array_equal(y, ref.astype(np.float32))


@pytest.mark.parametrize("stride", [1, 2])
def test_conv2d_vs_torch_f64(oracle_mod, stride):
    """Library special case: torch's float64 conv2d with padding 1 (cross-correlation)."""
    rng = np.random.default_rng(12)
    x = rng.uniform(-1, 1, (2, 7, 13, 10)).astype(np.float32)
    w = rng.normal(0, 0.2, (9, 7, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 9).astype(np.float32)
    y = oracle_mod.conv2d(x, w, b, stride=stride, act="none")
    ref = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                   torch.from_numpy(b).double(), stride=stride, padding=1).numpy()
    absref = F.conv2d(torch.from_numpy(np.abs(x)).double(), torch.from_numpy(np.abs(w)).double(),
                      torch.from_numpy(np.abs(b)).double(), stride=stride, padding=1).numpy()
    assert within_fp32_sum_bound(y, ref, absref, 9 * 7 + 1)


def test_conv3d_vs_torch_f64_causal(oracle_mod):
    """Library special case: conv3d over [carry, x] with padding (0,1,1) equals the causal conv."""
    rng = np.random.default_rng(13)
    x = rng.normal(0, 1, (1, 6, 5, 7, 9)).astype(np.float32)
    c = rng.normal(0, 1, (1, 6, 2, 7, 9)).astype(np.float32)
    w = rng.normal(0, 0.1, (4, 6, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 4).astype(np.float32)
    y = oracle_mod.conv3d_causal(x, w, b, carry=c)
    seq = torch.from_numpy(np.concatenate([c, x], axis=2)).double()
    ref = F.conv3d(seq, torch.from_numpy(w).double(), torch.from_numpy(b).double(),
                   padding=(0, 1, 1)).numpy()
    absref = F.conv3d(seq.abs(), torch.from_numpy(np.abs(w)).double(),
                      torch.from_numpy(np.abs(b)).double(), padding=(0, 1, 1)).numpy()
    assert within_fp32_sum_bound(y, ref, absref, 27 * 6 + 1)
    # first pass: zero history equals torch's front padding of 2 frames
    y0 = oracle_mod.conv3d_causal(x, w, b, carry=None)
    ref0 = F.conv3d(F.pad(torch.from_numpy(x).double(), (1, 1, 1, 1, 2, 0)),
                    torch.from_numpy(w).double(), torch.from_numpy(b).double()).numpy()
    assert np.max(np.abs(y0 - ref0)) < 1e-4


def test_layouts_agree(oracle_mod):
    rng = np.random.default_rng(14)
    x = rng.normal(0, 1, (1, 4, 3, 5, 6)).astype(np.float32)
    c = rng.normal(0, 1, (1, 4, 2, 5, 6)).astype(np.float32)
    w = rng.normal(0, 0.2, (3, 4, 3, 3, 3)).astype(np.float32)
    y1 = oracle_mod.conv3d_causal(x, w, None, carry=c)
    y2 = oracle_mod.conv3d_causal(x.transpose(0, 2, 3, 4, 1), w, None,
                                  carry=c.transpose(0, 2, 3, 4, 1), layout="NDHWC")
    assert np.array_equal(y1, y2.transpose(0, 4, 1, 2, 3))
    x2 = x[:, :, 0]
    w2 = w[:, :, 1]
    assert np.array_equal(oracle_mod.conv2d(x2, w2),
                          oracle_mod.conv2d(x2.transpose(0, 2, 3, 1), w2, layout="NHWC").transpose(0, 3, 1, 2))


# ------------------------------------------------------------------ invariants

def test_identity_and_delta_kernels(oracle_mod):
    rng = np.random.default_rng(15)
    x = rng.uniform(-1, 1, (1, 3, 6, 7)).astype(np.float32)
    b = np.array([0.5, -0.25, 0.0], np.float32)
    w = np.zeros((3, 3, 3, 3), np.float32)
    for c in range(3):
        w[c, c, 1, 1] = 1
    y = oracle_mod.conv2d(x, w, b)
    assert np.array_equal(y, x + b[None, :, None, None])
    # off-centre delta (kh=2, kw=0): y[h, w] = x[h+1, w-1], zero filled
    w = np.zeros((3, 3, 3, 3), np.float32)
    for c in range(3):
        w[c, c, 2, 0] = 1
    y = oracle_mod.conv2d(x, w)
    ref = np.zeros_like(x)
    ref[:, :, :-1, 1:] = x[:, :, 1:, :-1]
    assert np.array_equal(y, ref)
    # 3D: current-frame delta reproduces x; oldest-frame delta returns the carried frames first
    x3 = rng.normal(0, 1, (1, 2, 4, 3, 5)).astype(np.float32)
    c3 = rng.normal(0, 1, (1, 2, 2, 3, 5)).astype(np.float32)
    w3 = np.zeros((2, 2, 3, 3, 3), np.float32)
    for c in range(2):
        w3[c, c, 2, 1, 1] = 1
    assert np.array_equal(oracle_mod.conv3d_causal(x3, w3, carry=c3), x3)
    w3 = np.zeros((2, 2, 3, 3, 3), np.float32)
    for c in range(2):
        w3[c, c, 0, 1, 1] = 1
    y3 = oracle_mod.conv3d_causal(x3, w3, carry=c3)
    assert np.array_equal(y3, np.concatenate([c3, x3[:, :, :2]], axis=2))


def test_zero_padding_invariant(oracle_mod):
    """conv(x) equals the interior of conv over x embedded in an explicit ring of zeros."""
    rng = np.random.default_rng(16)
    x = rng.uniform(-1, 1, (1, 4, 8, 9)).astype(np.float32)
    w = rng.normal(0, 0.3, (5, 4, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 5).astype(np.float32)
    xp = np.zeros((1, 4, 10, 11), np.float32)
    xp[:, :, 1:-1, 1:-1] = x
    y = oracle_mod.conv2d(x, w, b)
    yp = oracle_mod.conv2d(xp, w, b)
    assert np.array_equal(y, yp[:, :, 1:-1, 1:-1])


def test_stride2_is_subsampled_stride1(oracle_mod):
    rng = np.random.default_rng(17)
    for H, W in ((8, 8), (7, 9), (1, 5)):
        x = rng.uniform(-1, 1, (2, 3, H, W)).astype(np.float32)
        w = rng.normal(0, 0.3, (4, 3, 3, 3)).astype(np.float32)
        b = rng.uniform(-0.1, 0.1, 4).astype(np.float32)
        y1 = oracle_mod.conv2d(x, w, b, stride=1, act="relu")
        y2 = oracle_mod.conv2d(x, w, b, stride=2, act="relu")
        assert np.array_equal(y2, y1[:, :, ::2, ::2])


def test_causality(oracle_mod):
    rng = np.random.default_rng(18)
    x = rng.normal(0, 1, (1, 3, 5, 4, 4)).astype(np.float32)
    w = rng.normal(0, 0.2, (2, 3, 3, 3, 3)).astype(np.float32)
    y = oracle_mod.conv3d_causal(x, w)
    for t in range(4):
        x2 = x.copy()
        x2[:, :, t + 1:] = rng.normal(0, 1, x2[:, :, t + 1:].shape)
        y2 = oracle_mod.conv3d_causal(x2, w)
        assert np.array_equal(y2[:, :, :t + 1], y[:, :, :t + 1])
        assert not np.array_equal(y2[:, :, t + 1:], y[:, :, t + 1:])


def test_chunking_with_carry_equals_one_pass(oracle_mod):
    """Two passes of 4 frames with the carried last two input frames equal one pass of 8."""
    rng = np.random.default_rng(19)
    x = rng.normal(0, 1, (1, 3, 8, 5, 6)).astype(np.float32)
    w = rng.normal(0, 0.2, (4, 3, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 4).astype(np.float32)
    full = oracle_mod.conv3d_causal(x, w, b)
    p1 = oracle_mod.conv3d_causal(x[:, :, :4], w, b)
    p2 = oracle_mod.conv3d_causal(x[:, :, 4:], w, b, carry=x[:, :, 2:4])
    assert np.array_equal(np.concatenate([p1, p2], axis=2), full)
    # and through a two-layer chain with per-layer carries
    layers = [dict(w=w, b=b, act="relu"),
              dict(w=rng.normal(0, 0.2, (2, 4, 3, 3, 3)).astype(np.float32), b=None)]
    yf, _ = oracle_mod.conv3d_chain(x, layers)
    y1, c1 = oracle_mod.conv3d_chain(x[:, :, :4], layers)
    y2, _ = oracle_mod.conv3d_chain(x[:, :, 4:], layers, carries=c1)
    assert np.array_equal(np.concatenate([y1, y2], axis=2), yf)


def test_unpatchify_is_a_bijection(oracle_mod):
    N, D, H, W = 1, 2, 3, 4
    y12 = np.arange(N * 12 * D * H * W, dtype=np.float32).reshape(N, 12, D, H, W)
    rgb = oracle_mod.unpatchify2x2(y12)
    assert rgb.shape == (N, 3, D, 2 * H, 2 * W)
    assert np.array_equal(np.sort(rgb.ravel()), np.sort(y12.ravel()))
    # c12 = rgb*4 + dy*2 + dx
    assert rgb[0, 2, 1, 2 * 1 + 1, 2 * 3 + 0] == y12[0, 2 * 4 + 1 * 2 + 0, 1, 1, 3]


def test_act_commutes_with_rounding(oracle_mod):
    """ReLU and clamp[-1,1] commute with round-to-nearest (monotone; 0 and +-1 representable)."""
    rng = np.random.default_rng(20)
    v = (rng.standard_normal(50000) * 2).astype(np.float32)
    for dt in ("f16", "bf16"):
        r, _ = oracle_mod.round_to(v, dt)
        a, _ = oracle_mod.round_to(np.maximum(v, 0), dt)
        assert np.array_equal(np.maximum(r, 0), a)
        a, _ = oracle_mod.round_to(np.clip(v, -1, 1), dt)
        assert np.array_equal(np.clip(r, -1, 1), a)


# ------------------------------------------------------------------ two-pass head (the page's split)

def test_head_split_identity(oracle_mod):
    """Without the early rounding, the temporal pass plus the nine shifted spatial sums equal the
    direct 27-tap convolution (within the fp32 summation bound, against float64 brute force)."""
    rng = np.random.default_rng(21)
    x = rng.normal(0, 1, (1, 5, 3, 4, 6)).astype(np.float32)
    c = rng.normal(0, 1, (1, 5, 2, 4, 6)).astype(np.float32)
    w = rng.normal(0, 0.2, (12, 5, 3, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.05, 0.05, 12).astype(np.float32)
    y2 = oracle_mod.head_two_pass(x, w, b, carry=c, round_g=False)
    ref, absref = brute_conv3d_f64(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64),
                                   c.astype(np.float64), "clamp")
    assert within_fp32_sum_bound(y2, ref, absref, 27 * 5 + 10)


def test_head_two_pass_exact_when_g_is_representable(oracle_mod):
    """Integer data whose temporal partial sums fit bf16's 8-bit significand: the early rounding is
    exact and both forms give the same values."""
    rng = np.random.default_rng(22)
    x = rng.integers(-1, 2, (1, 6, 2, 5, 7)).astype(np.float32)
    c = rng.integers(-1, 2, (1, 6, 2, 5, 7)).astype(np.float32)
    w = rng.choice([-1.0, 0.0, 1.0], size=(12, 6, 3, 3, 3), p=[0.1, 0.8, 0.1]).astype(np.float32)
    y2 = oracle_mod.head_two_pass(x, w, np.zeros(12, np.float32), carry=c)
    y1 = oracle_mod.conv3d_causal(x, w, np.zeros(12, np.float32), carry=c, act="clamp")
    assert np.array_equal(y2, y1)


def test_head_two_pass_rounds_g_before_the_spatial_sum(oracle_mod):
    """Hand-worked: one pixel, one channel path; the temporal sum g = 257 is not a bf16 value and
    rounds to 256 (ties to even), so with bias -256.5 the output is clamp(-0.5) = -0.5, where the
    one-accumulator form gives clamp(0.5) = 0.5."""
    x = np.zeros((1, 1, 1, 1, 1), np.float32)
    x[0, 0, 0, 0, 0] = 257.0
    w = np.zeros((12, 1, 3, 3, 3), np.float32)
    w[0, 0, 2, 1, 1] = 1.0          # output channel 0, current frame, centre tap
    b = np.zeros(12, np.float32)
    b[0] = -256.5
    assert oracle_mod.head_two_pass(x, w, b)[0, 0, 0, 0, 0] == -0.5
    assert oracle_mod.head_two_pass(x, w, b, round_g=False)[0, 0, 0, 0, 0] == 0.5
    assert oracle_mod.conv3d_causal(x, w, b, act="clamp")[0, 0, 0, 0, 0] == 0.5


# ------------------------------------------------------------------ banding (locality of the definition)

@pytest.mark.parametrize("dims", [2, 3])
def test_bands_with_halo_concatenate_to_the_plane(dims, oracle_mod):
    """Output rows depend only on input rows one above and one below (pad 1, 3 taps): the oracle run on a
    band's rows plus its halo rows (where they exist), with the rows it computes from its own zero padding
    dropped, gives exactly the whole plane's rows; concatenated bands equal the plane bit for bit. This is
    the banded mode's definition (FastVideo head.cu page: bands with their own row offset and the global
    height)."""
    oracle = oracle_mod
    rng = np.random.default_rng(8301 + dims)
    H, W = 17, 9
    if dims == 2:
        x = rng.integers(-2, 3, (2, 3, H, W)).astype(np.float32)
        w = rng.integers(-2, 3, (4, 3, 3, 3)).astype(np.float32)
        full = oracle.conv2d(x, w, None, act="relu")
        ax = 2
        run = lambda xs: oracle.conv2d(xs, w, None, act="relu")
    else:
        x = rng.integers(-2, 3, (1, 3, 2, H, W)).astype(np.float32)
        c = rng.integers(-2, 3, (1, 3, 2, H, W)).astype(np.float32)
        w = rng.integers(-2, 3, (4, 3, 3, 3, 3)).astype(np.float32)
        full = oracle.conv3d_causal(x, w, None, carry=c, act="relu")
        ax = 3
        run = None
    parts = []
    for lo, rows in [(0, 5), (5, 7), (12, 5)]:
        in_lo, in_hi = max(lo - 1, 0), min(lo + rows + 1, H)
        xs = np.take(x, range(in_lo, in_hi), axis=ax)
        if dims == 2:
            y = run(xs)
        else:
            y = oracle.conv3d_causal(xs, w, None, carry=np.take(c, range(in_lo, in_hi), axis=ax), act="relu")
        parts.append(np.take(y, range(lo - in_lo, lo - in_lo + rows), axis=ax))
    assert np.array_equal(np.concatenate(parts, axis=ax), full)
    # a band without its lower halo row differs (the halo is needed)
    xs = np.take(x, range(4, 11), axis=ax)
    y = run(xs) if dims == 2 else oracle.conv3d_causal(xs, w, None, carry=np.take(c, range(4, 11), axis=ax), act="relu")
    assert not np.array_equal(np.take(y, range(1, 7), axis=ax), np.take(full, range(5, 11), axis=ax))
