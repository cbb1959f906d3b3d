"""The environment switches that change a kernel's tile order, its form or the launch sequence give the
default path's values (include/x3conv.h lists them: the results are the same under every setting).

* X3CONV_FRAME_PAIRS=0: causal channels-last layers over an even number of frames compute their frames
  one after the other instead of in pairs: the same tiles and sums, so bit for bit the same output.
* X3CONV_TK=0: 8-channel channels-last layers leave the taps-in-K form for the horizontal-taps-in-N
  form; other fp32 sums, so both are compared with the oracle on integer data (exact).
* X3CONV_PDL=0: no programmatic dependent launches (carry copies on the side stream, layers fully
  serialised). The library reads it once per process, so a child process runs a two-pass causal stack
  with carries and a 2D NCHW stack with it set, and its outputs must equal this process's bit for bit
  on random data.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import assert_exact, dev, host_values

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


@pytest.mark.parametrize("variant", ["int", "random"])
def test_frame_pairs_off(variant, monkeypatch):
    D, H, W, C = 4, 20, 70, 128
    x = synth.activation([7100, 0], (1, D, H, W, C), "bf16", variant, ("normal", 1.0))
    carry = synth.activation([7100, 3], (1, 2, H, W, C), "bf16", variant, ("normal", 1.0))
    L = synth.make_layer([7100], 3, C, C, "bf16", act="relu", variant=variant)
    conv = x3.Conv(x3.make_desc(3, 1, C, C, H, W, D=D, act="relu"), dev(L.w), dev(L.b))
    assert conv.kernel_name == "igemm_tcgen05_sw128"
    y_pairs = host_values(conv(dev(x), dev(carry)), "bf16")
    monkeypatch.setenv("X3CONV_FRAME_PAIRS", "0")
    y_single = host_values(conv(dev(x), dev(carry)), "bf16")
    torch.cuda.synchronize()
    assert np.array_equal(y_pairs, y_single)
    if variant == "int":  # |partial sums| <= 128 * 27 * 2 * 2 + 2 < 2^24
        ref = oracle.conv3d_causal(x.vals, L.w.vals, L.b.vals, carry=carry.vals, act="relu", layout="NDHWC")
        assert_exact(y_single, ref, "bf16")


@pytest.mark.parametrize("case", [(4, 64, 37, 95, "relu"), (1, 24, 9, 31, "none")], ids=str)
def test_taps_in_k_off(case, monkeypatch):
    N, Co, H, W, act = case
    x = synth.activation([7200, 0], (N, H, W, 8), "f16", "int")
    L = synth.make_layer([7200, Co], 2, 8, Co, "f16", act=act, variant="int")

    def run():
        conv = x3.Conv(x3.make_desc(2, N, 8, Co, H, W, layout="NHWC", dtype="f16", act=act), dev(L.w), dev(L.b))
        return host_values(conv(dev(x)), "f16"), x3.conv_plan_describe(conv.plan)

    y_tk, g_tk = run()
    monkeypatch.setenv("X3CONV_TK", "0")
    y_tn, g_tn = run()
    torch.cuda.synchronize()
    assert g_tk["tn"] == 1 and g_tk["tk"] == 1
    assert g_tn["tn"] == 1 and g_tn["tk"] == 0
    ref = oracle.conv2d(x.vals, L.w.vals, L.b.vals, act=act, layout="NHWC")
    assert_exact(y_tk, ref, "f16")
    assert_exact(y_tn, ref, "f16")


def stacks_outputs():
    """Raw output bits of a causal 96 -> 128 -> 128 stack over two passes of 4 frames (carries written
    by the first pass and read by the second; the channels-last engine, carry copies as dependent
    kernels when dependent launches are on) and of a 2D NCHW f16 stack with a stride-2 layer (activations
    channels-last between the layers), random data."""
    out = {}
    chans, H, W = [96, 128, 128], 10, 100
    layers = [synth.make_layer([7300, i], 3, chans[i], chans[i + 1], "bf16", act=("relu", "none")[i])
              for i in range(2)]
    convs = [x3.Conv(x3.make_desc(3, 1, L.C_in, L.C_out, H, W, D=4, act=L.act), dev(L.w), dev(L.b))
             for L in layers]
    stack = x3.ConvStack(convs)
    x = dev(synth.activation([7300, 0], (1, 8, H, W, chans[0]), "bf16", "random", ("normal", 1.0)))
    carries = [torch.zeros((1, 2, H, W, c), dtype=torch.bfloat16, device="cuda") for c in chans[:-1]]
    ya = stack(x[:, :4].contiguous(), carries=carries, carry_valid=False)
    yb = stack(x[:, 4:].contiguous(), carries=carries, carry_valid=True)
    torch.cuda.synchronize()
    out["causal"] = torch.cat([ya, yb], dim=1).view(torch.int16).cpu().numpy()
    out["carries"] = np.concatenate([c.view(torch.int16).cpu().numpy().ravel() for c in carries])
    spec, N, h, w = [(3, 32, 1), (32, 32, 1), (32, 32, 2), (32, 32, 1)], 2, 40, 72
    layers2 = [synth.make_layer([7310, i], 2, ci, co, "f16", stride=s, act="relu") for i, (ci, co, s) in enumerate(spec)]
    convs2 = []
    for L in layers2:
        convs2.append(x3.Conv(x3.make_desc(2, N, L.C_in, L.C_out, h, w, stride=L.stride, dtype="f16", act="relu"),
                              dev(L.w), dev(L.b)))
        h, w = convs2[-1].H_out, convs2[-1].W_out
    x2 = dev(synth.activation([7310, 0], (N, 3, 40, 72), "f16", "random", ("uniform", -1.0, 1.0)))
    y2 = x3.ConvStack(convs2)(x2)
    torch.cuda.synchronize()
    out["nchw_stack"] = y2.view(torch.int16).cpu().numpy()
    return out


def save_stacks_outputs(path):
    """Child-process entry: load the library and write stacks_outputs() to `path` (.npz)."""
    x3.load()
    np.savez(path, **stacks_outputs())
    assert x3.conv_device_status(1) == x3.X3_OK


def test_dependent_launches_off(tmp_path):
    path = str(tmp_path / "pdl_off.npz")
    env = dict(os.environ, X3CONV_PDL="0")
    code = f"import sys; sys.path.insert(0, {ROOT!r}); import tests.test_gpu_switches as t; t.save_stacks_outputs({path!r})"
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    off = np.load(path)
    on = stacks_outputs()
    for k, v in on.items():
        assert np.array_equal(off[k], v), k
