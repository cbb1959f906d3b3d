"""GPU test of conv_stack_forward_noalloc, the stack driver for callers that must not allocate
device memory (for example a plug-in whose host framework owns every allocation): its
intermediate activations live in a buffer built into the library instead of a caller workspace.

It is called through the C ABI and compared bit for bit with conv_stack_forward (the workspace
version, the same plans and kernels) on the same layers, twice in a row with different inputs, so
that contents the shared buffer keeps from the first call cannot leak into the second. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024


def _noalloc_fn():
    lib = x3.load()
    fn = lib.conv_stack_forward_noalloc
    pp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [pp, ctypes.c_int, ctypes.c_void_p, pp, ctypes.c_int, pp, pp, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _arr(ptrs):
    a = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)), a


def _build(chans, D, H, W, seed):
    layers = [synth.make_layer([seed, i], 3, ci, co, "bf16", act="relu" if i + 2 < len(chans) else "none")
              for i, (ci, co) in enumerate(zip(chans[:-1], chans[1:]))]
    convs = [x3.Conv(x3.make_desc(3, 1, L.C_in, L.C_out, H, W, D=D, act=L.act), dev(L.w), dev(L.b))
             for L in layers]
    return convs


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def test_noalloc_matches_workspace_stack_twice():
    chans, D, H, W = [32, 48, 64, 16], 3, 9, 140
    convs = _build(chans, D, H, W, 5100)
    stack = x3.ConvStack(convs)
    assert 0 < stack.ws_bytes <= SCRATCH_BYTES
    fn = _noalloc_fn()
    plans, k1 = _arr([c.plan for c in convs])
    wts, k2 = _arr([c._wp for c in convs])
    bias, k3 = _arr([c.bias.data_ptr() for c in convs])
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        x = dev(synth.activation([5100, 10 + call], (1, D, H, W, 32), "bf16", "random", ("normal", 1.0)))
        hist = [dev(synth.activation([5100, 20 + call, i], (1, 2, H, W, c), "bf16", "random", ("normal", 1.0)))
                for i, c in enumerate(chans[:-1])]
        c_ref = [h.clone() for h in hist]
        c_new = [h.clone() for h in hist]
        y_ref = stack(x, carries=c_ref, carry_valid=True)
        y_new = torch.empty_like(y_ref)
        cp, k4 = _arr([c.data_ptr() for c in c_new])
        st = fn(plans, len(convs), x.data_ptr(), cp, 1, wts, bias, y_new.data_ptr(), stream)
        assert st == x3.X3_OK, x3.conv_last_error()
        torch.cuda.synchronize()
        # the same plans and kernels as the workspace version: the values must agree bit for bit (a
        # tolerance would hide a stale part of the shared scratch)
        assert torch.equal(y_new, y_ref)
        for a, b in zip(c_new, c_ref):
            assert torch.equal(a, b)


def test_noalloc_matches_workspace_channels_last_2d_stack():
    """A TAESD-like 2D NCHW stack (kept channels-last between its layers, stride 2 inside, NCHW out):
    the built-in scratch holds the converted input and the ping-pong activations; twice in a row,
    bit for bit the workspace version."""
    N, H, W = 1, 96, 128
    spec = [(3, 64, 1), (64, 64, 1), (64, 64, 2), (64, 64, 1)]
    layers = [synth.make_layer([5200, i], 2, ci, co, "f16", stride=s, act="relu")
              for i, (ci, co, s) in enumerate(spec)]
    convs, h, w = [], H, W
    for L in layers:
        convs.append(x3.Conv(x3.make_desc(2, N, L.C_in, L.C_out, h, w, stride=L.stride, dtype="f16", act="relu"),
                             dev(L.w), dev(L.b)))
        h, w = convs[-1].H_out, convs[-1].W_out
    stack = x3.ConvStack(convs)
    assert 0 < stack.ws_bytes <= SCRATCH_BYTES
    fn = _noalloc_fn()
    plans, k1 = _arr([c.plan for c in convs])
    wts, k2 = _arr([c._wp for c in convs])
    bias, k3 = _arr([c.bias.data_ptr() for c in convs])
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        x = dev(synth.activation([5200, 10 + call], (N, 3, H, W), "f16", "random", ("uniform", -1.0, 1.0)))
        y_ref = stack(x)
        y_new = torch.empty_like(y_ref)
        st = fn(plans, len(convs), x.data_ptr(), None, 0, wts, bias, y_new.data_ptr(), stream)
        assert st == x3.X3_OK, x3.conv_last_error()
        torch.cuda.synchronize()
        assert torch.equal(y_new, y_ref)


def test_noalloc_rejects_stacks_beyond_its_scratch():
    # two 128-channel 4-frame 352x624 intermediates need far more than the built-in scratch
    convs = [x3.Conv(x3.make_desc(3, 1, 128, 128, 352, 624, D=4, act="relu"),
                     torch.zeros((128, 128, 3, 3, 3), dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(128, dtype=torch.bfloat16, device="cuda")) for _ in range(3)]
    assert x3.conv_stack_workspace_bytes([c.plan for c in convs]) > SCRATCH_BYTES
    fn = _noalloc_fn()
    plans, k1 = _arr([c.plan for c in convs])
    wts, k2 = _arr([c._wp for c in convs])
    bias, k3 = _arr([c.bias.data_ptr() for c in convs])
    st = fn(plans, 3, 16, None, 0, wts, bias, 4096, None)
    assert st == x3.X3_ERR_OOM
    assert "scratch" in x3.conv_last_error()
