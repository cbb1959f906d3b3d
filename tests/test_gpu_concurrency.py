"""Calls from several host threads on their own streams at once give the results of one thread.

The entry points keep no state between calls but the plan and the caller's buffers (and, per calling
thread and device, the side stream of conv_stack_forward), so two threads driving different layers on
different streams must get, on every one of many repetitions, the bits that one thread gets alone.
"""
import threading

import pytest
import torch

import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import synth
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x3.load()
    yield
    assert x3.conv_device_status(1) == x3.X3_OK


def test_two_threads_two_streams():
    # thread 0: a causal 128 -> 128 layer (channels-last engine) with its two carried frames
    D, H, W, C = 4, 40, 200, 128
    L3 = synth.make_layer([7400], 3, C, C, "bf16", act="relu")
    conv3 = x3.Conv(x3.make_desc(3, 1, C, C, H, W, D=D, act="relu"), dev(L3.w), dev(L3.b))
    x3d = dev(synth.activation([7400, 0], (1, D, H, W, C), "bf16", "random", ("normal", 1.0)))
    c3d = dev(synth.activation([7400, 3], (1, 2, H, W, C), "bf16", "random", ("normal", 1.0)))
    # thread 1: a 2D NCHW f16 stack 3 -> 32 -> 32 (stride 2) -> 32, channels-last between the layers
    N, h, w = 4, 96, 128
    convs, hh, ww = [], h, w
    for i, (ci, co, s) in enumerate([(3, 32, 1), (32, 32, 2), (32, 32, 1)]):
        L = synth.make_layer([7410, i], 2, ci, co, "f16", stride=s, act="relu")
        convs.append(x3.Conv(x3.make_desc(2, N, ci, co, hh, ww, stride=s, dtype="f16", act="relu"), dev(L.w), dev(L.b)))
        hh, ww = convs[-1].H_out, convs[-1].W_out
    stack2d = x3.ConvStack(convs)
    x2d = dev(synth.activation([7410, 0], (N, 3, h, w), "f16", "random", ("uniform", -1.0, 1.0)))

    want3 = conv3(x3d, c3d)
    want2 = stack2d(x2d)
    torch.cuda.synchronize()

    reps = 20
    outs3 = [torch.empty_like(want3) for _ in range(reps)]
    outs2 = [torch.empty_like(want2) for _ in range(reps)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    failures = []
    start = threading.Barrier(2)

    def run(k):
        try:
            torch.cuda.set_device(0)
            s = streams[k]
            start.wait()
            with torch.cuda.stream(s):
                for r in range(reps):
                    if k == 0:
                        conv3(x3d, c3d, out=outs3[r], stream=s)
                    else:
                        stack2d(x2d, out=outs2[r], stream=s)
            s.synchronize()
        except Exception as e:  # reported by the main thread
            failures.append((k, repr(e)))

    threads = [threading.Thread(target=run, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not failures, failures
    for r in range(reps):
        assert torch.equal(outs3[r].view(torch.int16), want3.view(torch.int16)), f"causal layer, repetition {r}"
        assert torch.equal(outs2[r].view(torch.int16), want2.view(torch.int16)), f"2D stack, repetition {r}"
