"""Seeded synthetic inputs for the convolution workloads.

This module is shared by the CUDA-path tests, the oracle tests and the bench. It holds no
convolution arithmetic: it only draws numbers and stores them in the 16-bit storage types
(numpy's float16 cast and torch's bfloat16 cast, both round-to-nearest-even library routines),
and returns the raw 16-bit patterns (fed to the GPU) together with their exact float32 values
(fed to the oracle), so both sides consume identical inputs.

Distributions follow the decoder workloads: activations U[-1,1] (2D) or N(0,1) (3D), weights
N(0, 1/sqrt(taps*C_in)) (the second parameter read as the standard deviation), biases
U[-0.1,0.1] (U[-0.05,0.05] for the head), and an integer variant with every value in {-2..2}
("fewtaps": integer inputs and three +-1 weights per output channel, for exact long chains).
Keys are numpy SeedSequence([1000 + workload id, tensor id]).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

STORAGE = {"f16": torch.float16, "bf16": torch.bfloat16}


def _rng(key):
    if isinstance(key, int):
        key = [key]
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


def to_storage(values: np.ndarray, dtype: str):
    """float64/float32 values -> (uint16 bits, exact float32 values) of the storage type."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64)).to(STORAGE[dtype])
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    vals = t.to(torch.float32).numpy().copy()
    return bits, vals


def draw(key, shape, dist, dtype: str):
    """Draw one tensor. dist: ('uniform', lo, hi) | ('normal', std) | ('int', lo, hi)."""
    g = _rng(key)
    kind = dist[0]
    if kind == "uniform":
        v = g.uniform(dist[1], dist[2], size=shape)
    elif kind == "normal":
        v = g.normal(0.0, dist[1], size=shape)
    elif kind == "int":
        v = g.integers(dist[1], dist[2] + 1, size=shape).astype(np.float64)
    else:
        raise ValueError(kind)
    return to_storage(v, dtype)


@dataclasses.dataclass
class Tensor:
    bits: np.ndarray      # uint16 storage pattern, in the tensor's own layout
    vals: np.ndarray      # exact float32 values, same layout
    dtype: str

    @property
    def shape(self):
        return self.bits.shape

    def torch(self, device="cpu") -> torch.Tensor:
        t = torch.from_numpy(self.bits.view(np.int16).copy()).view(STORAGE[self.dtype])
        return t.to(device)


def tensor(key, shape, dist, dtype) -> Tensor:
    bits, vals = draw(key, shape, dist, dtype)
    return Tensor(bits, vals, dtype)


@dataclasses.dataclass
class Layer:
    """One convolution layer's parameters (canonical weight layout [C_out][C_in][(3)][3][3])."""
    dims: int
    C_in: int
    C_out: int
    stride: int
    act: str
    w: Tensor
    b: Tensor | None


def make_layer(key, dims, C_in, C_out, dtype, stride=1, act="none", variant="random",
               bias_range=0.1) -> Layer:
    taps = 9 if dims == 2 else 27
    wshape = (C_out, C_in) + (3,) * dims
    if variant == "int":
        w = tensor(list(key) + [1], wshape, ("int", -2, 2), dtype)
        b = tensor(list(key) + [2], (C_out,), ("int", -2, 2), dtype)
    elif variant == "sparse1":
        # weights in {-1,0,1}, mostly zero, and integer bias: keeps head sums inside [-1,1]
        g = _rng(list(key) + [1])
        v = g.choice([-1.0, 0.0, 1.0], size=wshape, p=[0.02, 0.96, 0.02])
        w = Tensor(*to_storage(v, dtype), dtype)
        b = tensor(list(key) + [2], (C_out,), ("int", 0, 0), dtype)
    elif variant == "fewtaps":
        # three non-zero weights (+1 or -1) per output channel at random (input channel, tap) places
        # and a bias in {-1, 0, 1}: every output is an integer sum of at most three inputs and the
        # bias, so a chain of many layers stays exact in fp32 and inside f16's range
        g = _rng(list(key) + [1])
        v = np.zeros(wshape)
        flat = v.reshape(C_out, -1)
        for co in range(C_out):
            flat[co, g.choice(flat.shape[1], size=min(3, flat.shape[1]), replace=False)] = g.choice([-1.0, 1.0], size=3)
        w = Tensor(*to_storage(v, dtype), dtype)
        b = tensor(list(key) + [2], (C_out,), ("int", -1, 1), dtype)
    else:
        std = 1.0 / np.sqrt(taps * C_in)
        w = tensor(list(key) + [1], wshape, ("normal", std), dtype)
        b = tensor(list(key) + [2], (C_out,), ("uniform", -bias_range, bias_range), dtype)
    return Layer(dims, C_in, C_out, stride, act, w, b)


def activation(key, shape, dtype, variant="random", dist=None) -> Tensor:
    if variant in ("int", "fewtaps"):
        return tensor(key, shape, ("int", -2, 2), dtype)
    if variant == "sparse1":
        return tensor(key, shape, ("int", -1, 1), dtype)
    return tensor(key, shape, dist, dtype)


# ------------------------------------------------------------------ decoder-shaped workloads

def conv2d_single(N=1, C=16, H=64, W=64, variant="random", seed=1001, C_out=None, stride=1,
                  act="relu", dtype="f16"):
    """One 2D NCHW conv (16->16, 64x64, bias + ReLU at full size)."""
    C_out = C if C_out is None else C_out
    x = activation([seed, 0], (N, C, H, W), dtype, variant, ("uniform", -1.0, 1.0))
    L = make_layer([seed], 2, C, C_out, dtype, stride=stride, act=act, variant=variant)
    return x, L


TAESD_CHAIN = [  # (C_in, C_out, stride): 3->64, 3x 64->64, 64->64 s2, 2x 64->64
    (3, 64, 1), (64, 64, 1), (64, 64, 1), (64, 64, 1), (64, 64, 2), (64, 64, 1), (64, 64, 1)]


def taesd_chain(N=4, H=256, W=256, variant="random", seed=1002, dtype="f16"):
    """TAESD-like chain of 2D NCHW convs, each with bias and ReLU."""
    x = activation([seed, 0], (N, 3, H, W), dtype, variant, ("uniform", -1.0, 1.0))
    layers = [make_layer([seed, 10 + i], 2, ci, co, dtype, stride=s, act="relu", variant=variant)
              for i, (ci, co, s) in enumerate(TAESD_CHAIN)]
    return x, layers


def conv3d_single(C_in=256, C_out=256, D=4, H=88, W=156, N=1, variant="random", seed=1003,
                  act="none", dtype="bf16", bias_range=0.1, with_carry=True):
    """One causal 3D NDHWC conv with 2 carried frames."""
    dist = ("normal", 1.0)
    x = activation([seed, 0], (N, D, H, W, C_in), dtype, variant, dist)
    carry = activation([seed, 3], (N, 2, H, W, C_in), dtype, variant, dist) if with_carry else None
    L = make_layer([seed], 3, C_in, C_out, dtype, act=act, variant=variant, bias_range=bias_range)
    return x, carry, L


def conv3d_stack(D=4, H=352, W=624, H3=176, W3=312, C=128, C3_in=256, variant="random",
                 seed=1004, dtype="bf16"):
    """Two chained C->C causal layers with ReLU, plus a 256->128 layer on its own input."""
    dist = ("normal", 1.0)
    x = activation([seed, 0], (1, D, H, W, C), dtype, variant, dist)
    carries = [activation([seed, 3, i], (1, 2, H, W, C), dtype, variant, dist) for i in range(2)]
    layers = [make_layer([seed, 10 + i], 3, C, C, dtype, act="relu", variant=variant) for i in range(2)]
    x3 = activation([seed, 20], (1, D, H3, W3, C3_in), dtype, variant, dist)
    carry3 = activation([seed, 23], (1, 2, H3, W3, C3_in), dtype, variant, dist)
    L3 = make_layer([seed, 12], 3, C3_in, C, dtype, act="none", variant=variant)
    return dict(x=x, carries=carries, layers=layers, x3=x3, carry3=carry3, L3=L3)


def head(D=4, H=352, W=624, C_in=256, variant="random", seed=1005, dtype="bf16", N=1):
    """conv_out head: causal 256->12 with clamp (bias U[-0.05,0.05])."""
    return conv3d_single(C_in=C_in, C_out=12, D=D, H=H, W=W, N=N, variant=variant, seed=seed,
                         act="clamp", dtype=dtype, bias_range=0.05)
