"""Full-size parity of the multi-layer workloads, in the launch configuration bench.py times.

* TAESD-like chain, N=4, 3x256x256, NCHW f16, 7 layers through conv_stack_forward: compared with
  the oracle run layer by layer with the library's rounding of each intermediate (full tensors).
* Decoder stack, two chained causal 128->128 layers at 4+2 x 352x624 through conv_stack_forward with
  carries: the stack's output equals the two layers run one by one through conv_forward bit for bit,
  and each layer matches the oracle on sampled positions (the second layer fed the first layer's
  GPU output), as does the carry the driver writes.
"""
import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_close, dev, host_values, oracle_sampled_3d, sample_positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def test_taesd_chain_full_size():
    xt, layers = synth.taesd_chain(seed=1002)
    convs, H, W = [], 256, 256
    for L in layers:
        d = x3.make_desc(2, 4, L.C_in, L.C_out, H, W, stride=L.stride, layout="NCHW", dtype="f16", act="relu")
        convs.append(x3.Conv(d, dev(L.w), dev(L.b)))
        H, W = convs[-1].H_out, convs[-1].W_out
    assert all(c.kernel_name.startswith("igemm_tcgen05") for c in convs)
    got = host_values(x3.ConvStack(convs)(dev(xt)), "f16")
    torch.cuda.synchronize()
    y = xt.vals
    for L in layers:
        y, _ = oracle.round_to(oracle.conv2d(y, L.w.vals, L.b.vals, stride=L.stride, act="relu"), "f16")
    assert got.shape == (4, 64, 128, 128)
    assert_close(got, y)
    ref32 = oracle.conv2d_chain(xt.vals, [dict(w=L.w.vals, b=L.b.vals, stride=L.stride, act="relu") for L in layers])
    assert_close(got, ref32)


def test_decoder_stack_full_size():
    st = synth.conv3d_stack(seed=1004)
    convs = [x3.Conv(x3.make_desc(3, 1, 128, 128, 352, 624, D=4, act=L.act), dev(L.w), dev(L.b))
             for L in st["layers"]]
    stack = x3.ConvStack(convs)
    x = dev(st["x"])
    c_stack = [dev(c).contiguous() for c in st["carries"]]
    c_ref = [c.clone() for c in c_stack]
    y_stack = stack(x, carries=c_stack, carry_valid=True)
    y1 = convs[0](x, c_ref[0])
    y2 = convs[1](y1, c_ref[1])
    torch.cuda.synchronize()
    assert torch.equal(y_stack, y2)
    # the driver's new carries: the last two frames of each layer's input sequence
    assert torch.equal(c_stack[0], x[:, 2:4])
    assert torch.equal(c_stack[1], y1[:, 2:4])
    pos = sample_positions(4, 352, 624, 300, seed=11)
    for i, (inp, carry, out) in enumerate(((x, c_ref[0], y1), (y1, c_ref[1], y2))):
        L = st["layers"][i]
        seq = np.concatenate([host_values(carry, "bf16"), host_values(inp, "bf16")], axis=1)
        ref = oracle_sampled_3d(seq, L.w.vals, L.b.vals, L.act, pos)
        o = host_values(out, "bf16")
        assert_close(np.stack([o[0, t, h, w] for (t, h, w) in pos]), ref)
