"""GPU tests of conv_stack_forward: chained layers through the caller's workspace, the causal
per-layer carries, and passes of a few frames that reproduce one long pass.

Expected values: the oracle run layer by layer, each layer's output rounded once to the storage
type before it feeds the next layer (the library stores every intermediate in bf16/f16). On
integer-valued data every fp32 sum is exact, so the comparison is bit for bit; on random data the
stack is also compared with the oracle's all-fp32 chain within the relative tolerances.
"""
import numpy as np
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


def make_3d_layers(chans, acts, variant, seed):
    return [synth.make_layer([seed, i], 3, ci, co, "bf16", act=a, variant=variant)
            for i, ((ci, co), a) in enumerate(zip(zip(chans[:-1], chans[1:]), acts))]


def oracle_rounded_chain_3d(x, carries, layers, dtype="bf16"):
    """Layer-by-layer oracle with the intermediate rounding the library applies; returns the
    final output (fp32 values, rounded) and each layer's input sequence's last two frames."""
    y = x
    new_carries = []
    for i, L in enumerate(layers):
        c = None if carries is None else carries[i]
        seq = y if c is None else np.concatenate([c, y], axis=1)
        new_carries.append(seq[:, -2:].copy())
        out = oracle.conv3d_causal(y, L.w.vals, L.b.vals, carry=c, act=L.act, layout="NDHWC")
        y, _ = oracle.round_to(out, dtype)
    return y, new_carries


def build_stack(layers, D, H, W):
    convs = [x3.Conv(x3.make_desc(3, 1, L.C_in, L.C_out, H, W, D=D, act=L.act), dev(L.w), dev(L.b))
             for L in layers]
    return convs, x3.ConvStack(convs)


@pytest.mark.parametrize("variant", ["int", "random"])
def test_stack3d_matches_layerwise_oracle(variant):
    # integer data: two layers keep every fp32 partial sum below 2^24 (27*48*2*3458 < 2^24)
    chans, acts = ([32, 48, 16], ["relu", "none"]) if variant == "int" else ([32, 48, 64, 16], ["relu", "relu", "none"])
    D, H, W = 3, 9, 140
    layers = make_3d_layers(chans, acts, variant, 4100)
    x = synth.activation([4100, 0], (1, D, H, W, 32), "bf16", variant, ("normal", 1.0))
    carries = [synth.activation([4100, 3, i], (1, 2, H, W, c), "bf16", variant, ("normal", 1.0))
               for i, c in enumerate(chans[:-1])]
    convs, stack = build_stack(layers, D, H, W)
    widest = max(chans[1:-1])
    n_buf = 2 if len(layers) > 2 else 1
    assert stack.ws_bytes == n_buf * ((1 * D * H * W * widest * 2 + 255) // 256 * 256)
    cdev = [dev(c).contiguous() for c in carries]
    y = stack(dev(x), carries=cdev, carry_valid=True)
    torch.cuda.synchronize()
    got = host_values(y, "bf16")
    want, want_carries = oracle_rounded_chain_3d(x.vals, [c.vals for c in carries], layers)
    if variant == "int":
        assert_exact(got, want, "bf16")
    else:
        assert_close(got, want)
        ref32, _ = oracle.conv3d_chain(x.vals, [dict(w=L.w.vals, b=L.b.vals, act=L.act) for L in layers],
                                       carries=[c.vals for c in carries], layout="NDHWC")
        assert_close(got, ref32)
    # every carry now holds the last two frames of its layer's input sequence (for layers past the
    # first that input is an intermediate, equal to the oracle's only within tolerance on random data)
    for i, c in enumerate(cdev):
        if variant == "int" or i == 0:
            assert np.array_equal(host_values(c, "bf16"), want_carries[i])
        else:
            assert_close(host_values(c, "bf16"), want_carries[i])


def test_stack3d_passes_equal_one_long_pass():
    """Two passes of 4 frames (zero history, then the carried frames) give the frames that one
    8-frame pass gives; integer data, so the comparison is exact."""
    chans, acts = [16, 32, 16], ["relu", "none"]
    H, W = 6, 130
    layers = make_3d_layers(chans, acts, "int", 4200)
    x = synth.activation([4200, 0], (1, 8, H, W, 16), "bf16", "int")
    convs8, stack8 = build_stack(layers, 8, H, W)
    y8 = host_values(stack8(dev(x)), "bf16")
    convs4, stack4 = build_stack(layers, 4, H, W)
    cdev = [torch.full((1, 2, H, W, c), 7.0, dtype=torch.bfloat16, device="cuda") for c in chans[:-1]]
    xd = dev(x)
    ya = host_values(stack4(xd[:, :4].contiguous(), carries=cdev, carry_valid=False), "bf16")
    yb = host_values(stack4(xd[:, 4:].contiguous(), carries=cdev, carry_valid=True), "bf16")
    torch.cuda.synchronize()
    assert np.array_equal(np.concatenate([ya, yb], axis=1), y8)
    want, _ = oracle_rounded_chain_3d(x.vals, None, layers)
    assert_exact(y8, want, "bf16")


def test_stack3d_single_frame_passes():
    """D = 1: the new history is [previous history frame 1, the input frame]."""
    chans, acts = [8, 16], ["none"]
    H, W = 5, 24
    layers = make_3d_layers(chans, acts, "int", 4300)
    x = synth.activation([4300, 0], (1, 3, H, W, 8), "bf16", "int")
    conv = x3.Conv(x3.make_desc(3, 1, 8, 16, H, W, D=1), dev(layers[0].w), dev(layers[0].b))
    stack = x3.ConvStack([conv])
    c = torch.zeros((1, 2, H, W, 8), dtype=torch.bfloat16, device="cuda")
    xd = dev(x)
    outs = [host_values(stack(xd[:, t:t + 1].contiguous(), carries=[c], carry_valid=t > 0), "bf16")
            for t in range(3)]
    want, _ = oracle_rounded_chain_3d(x.vals, None, layers)
    assert_exact(np.concatenate(outs, axis=1), want, "bf16")


TAESD_LIKE = {
    # integer data: two layers stay inside f16's range (16*9*2*110 < 65504) with exact fp32 sums
    "int": [(3, 16, 1), (16, 16, 2)],
    # {-1,0,1} data, sparse weights: small exact sums through four layers, stride 2 inside the chain
    "sparse1": [(3, 16, 1), (16, 16, 1), (16, 16, 2), (16, 8, 1)],
    "random": [(3, 32, 1), (32, 32, 1), (32, 32, 2), (32, 32, 1)],
}


@pytest.mark.parametrize("layout", ["channels_last", "nchw"])
@pytest.mark.parametrize("variant", ["int", "sparse1", "random"])
def test_stack2d_taesd_like(variant, layout, monkeypatch):
    """A shortened TAESD-like chain at reduced size, NCHW f16 in and out. channels_last: the driver
    keeps the activations between layers channels-last (the default when every layer has that form
    and the last one has stride 1); nchw: every layer runs its own NCHW form."""
    if layout == "nchw":
        monkeypatch.setenv("X3CONV_STACK_LAYOUT", "nchw")
    N, H, W = 2, 40, 72
    spec = TAESD_LIKE[variant]
    x = synth.activation([4400, 0], (N, 3, H, W), "f16", variant, ("uniform", -1.0, 1.0))
    layers = [synth.make_layer([4400, i], 2, ci, co, "f16", stride=s, act="relu", variant=variant)
              for i, (ci, co, s) in enumerate(spec)]
    convs, h, w = [], H, W
    for L in layers:
        convs.append(x3.Conv(x3.make_desc(2, N, L.C_in, L.C_out, h, w, stride=L.stride, dtype="f16", act="relu"),
                             dev(L.w), dev(L.b)))
        h, w = convs[-1].H_out, convs[-1].W_out
    stack = x3.ConvStack(convs)
    got = host_values(stack(dev(x)), "f16")
    torch.cuda.synchronize()
    y = x.vals
    for L in layers:
        y, _ = oracle.round_to(oracle.conv2d(y, L.w.vals, L.b.vals, stride=L.stride, act="relu"), "f16")
    if variant != "random":
        assert np.array_equal(got, y)
    else:
        assert_close(got, y)
        ref32 = oracle.conv2d_chain(x.vals, [dict(w=L.w.vals, b=L.b.vals, stride=L.stride, act="relu")
                                             for L in layers])
        assert_close(got, ref32)


def test_stack3d_wide_channels():
    """Chained 64->128->128 layers: the 128-channel layers run on the swapped-operand engine."""
    chans, acts = [64, 128, 128], ["relu", "none"]
    D, H, W = 2, 6, 140
    layers = make_3d_layers(chans, acts, "random", 4500)
    x = synth.activation([4500, 0], (1, D, H, W, 64), "bf16", "random", ("normal", 1.0))
    carries = [synth.activation([4500, 3, i], (1, 2, H, W, c), "bf16", "random", ("normal", 1.0))
               for i, c in enumerate(chans[:-1])]
    convs, stack = build_stack(layers, D, H, W)
    assert all(c.kernel_name == "igemm_tcgen05_sw128" for c in convs)
    cdev = [dev(c).contiguous() for c in carries]
    got = host_values(stack(dev(x), carries=cdev, carry_valid=True), "bf16")
    torch.cuda.synchronize()
    want, want_carries = oracle_rounded_chain_3d(x.vals, [c.vals for c in carries], layers)
    assert_close(got, want)
    assert np.array_equal(host_values(cdev[0], "bf16"), want_carries[0])
    assert_close(host_values(cdev[1], "bf16"), want_carries[1])


def test_stack2d_layouts_agree_on_odd_shapes(monkeypatch):
    """Channel counts that are not multiples of 64, odd sizes, stride 2 with odd input sizes, one
    image: the channels-last stack against the per-layer NCHW stack and the oracle."""
    N, H, W = 1, 37, 83
    spec = [(5, 24, 1), (24, 40, 2), (40, 72, 1), (72, 136, 1), (136, 16, 1)]
    x = synth.activation([4600, 0], (N, 5, H, W), "bf16", "random", ("uniform", -1.0, 1.0))
    layers = [synth.make_layer([4600, i], 2, ci, co, "bf16", stride=s, act="relu" if i < 4 else "none")
              for i, (ci, co, s) in enumerate(spec)]
    convs, h, w = [], H, W
    for L in layers:
        convs.append(x3.Conv(x3.make_desc(2, N, L.C_in, L.C_out, h, w, stride=L.stride, dtype="bf16", act=L.act),
                             dev(L.w), dev(L.b)))
        h, w = convs[-1].H_out, convs[-1].W_out
    assert all("shadow" in x3.conv_plan_describe(c.plan) for c in convs)
    y_cl = host_values(x3.ConvStack(convs)(dev(x)), "bf16")
    monkeypatch.setenv("X3CONV_STACK_LAYOUT", "nchw")
    y_nc = host_values(x3.ConvStack(convs)(dev(x)), "bf16")
    torch.cuda.synchronize()
    assert y_cl.shape == y_nc.shape == (1, 16, 19, 42)
    ref = x.vals
    for L in layers:
        ref, _ = oracle.round_to(oracle.conv2d(ref, L.w.vals, L.b.vals, stride=L.stride, act=L.act), "bf16")
    assert_close(y_cl, ref)
    assert_close(y_nc, ref)


@pytest.mark.parametrize("path", ["side_stream", "dependent_kernel"])
def test_stack3d_carry_copies_finish_within_the_call(path):
    """The carry copies are part of the call's work on the caller's stream: work the caller enqueues
    on that stream right after the call (here: overwriting the input, which the first layer's copy
    reads) must not reach a copy still reading it. Four layers, so the second layer's copy reads a
    workspace half that the third layer overwrites inside the call. Layers with fewer than 96 output
    channels run on engines whose copies go on the library's side stream; 96 or more run on the
    channels-last tensor-core engine, whose copies are kernels launched as programmatic dependents
    of the layer (random data there: the fp32 sums of wide integer layers are not exact)."""
    if path == "side_stream":
        chans, acts, variant = [64, 32, 32, 32, 16], ["relu", "relu", "relu", "none"], "int"
    else:
        chans, acts, variant = [96, 128, 128, 128, 96], ["relu", "relu", "relu", "none"], "random"
    D, H, W = 4, 24, 200
    layers = make_3d_layers(chans, acts, variant, 4700)
    x = synth.activation([4700, 1], (1, D, H, W, chans[0]), "bf16", variant, ("normal", 1.0))
    carries = [synth.activation([4700, 2, i], (1, 2, H, W, c), "bf16", variant, ("normal", 1.0))
               for i, c in enumerate(chans[:-1])]
    convs, stack = build_stack(layers, D, H, W)
    engines = {c.kernel_name for c in convs}
    assert all(n.startswith("igemm_tcgen05_sw128") for n in engines) == (path == "dependent_kernel"), engines
    side = torch.cuda.Stream()
    xd = dev(x)
    cdev = [dev(c).contiguous() for c in carries]
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        y = stack(xd, carries=cdev, carry_valid=True, stream=side)
        xd.fill_(0)  # same stream, right after the call
    torch.cuda.synchronize()
    want, want_carries = oracle_rounded_chain_3d(x.vals, [c.vals for c in carries], layers)
    # the first carry is a plain copy of the input's last two frames: exact on any data
    assert np.array_equal(host_values(cdev[0], "bf16"), want_carries[0]), "carry 0"
    if variant == "int":
        assert_exact(host_values(y, "bf16"), want, "bf16")
        for i, c in enumerate(cdev):
            assert np.array_equal(host_values(c, "bf16"), want_carries[i]), f"carry {i}"
    else:
        assert_close(host_values(y, "bf16"), want)
        for i, c in enumerate(cdev[1:], start=1):
            assert_close(host_values(c, "bf16"), want_carries[i])
