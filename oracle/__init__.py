"""CPU oracle for the 3x3 / causal 3x3x3 convolution hot path.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The product path (the CUDA library and the
``x3x3_convolution_gb300`` binding) never imports it, and this package imports nothing from the
product: the two share no code.

The arithmetic lives in ``x3conv_oracle.c`` (plain fp32 nested loops, built with
``-ffp-contract=off`` so that every multiply and add rounds separately, identically on x86 and
Arm). This module only marshals numpy arrays into it and does layout permutations.

Definitions followed (see the C file for the full list):
  * musetalk-bench ``patches/taesd_conv.cuh.new``, ``taesd_conv3x3_impl``: 2D pad-1 3x3
    cross-correlation, stride 1 or 2, bias-initialised fp32 accumulator, optional ReLU.
  * FastVideo ``wan22_vae_decode/solution/head.cu``, header comment and ``head_stencil_kernel``:
    causal 3x3x3 over [2 carried frames, current frames], all 27 taps in one fp32 accumulator,
    clamp to [-1,1], one rounding at the store.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "x3conv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_x3conv.so")

ACT = {"none": 0, "relu": 1, "clamp": 2}
DTYPE = {"f16": 0, "bf16": 1}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` with gcc (OpenMP, no FP contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def configure(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_conv2d.argtypes = [f32p, f32p, f32p, f32p] + [ctypes.c_int] * 8
    lib.oracle_conv2d.restype = ctypes.c_int
    lib.oracle_conv3d_causal.argtypes = [f32p, f32p, f32p, f32p, f32p] + [ctypes.c_int] * 8
    lib.oracle_conv3d_causal.restype = ctypes.c_int
    lib.oracle_round_to.argtypes = [f32p, f32p, ctypes.c_size_t, ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_uint16)]
    lib.oracle_round_to.restype = None
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_unpatchify2x2.argtypes = [f32p, f32p] + [ctypes.c_int] * 4
    lib.oracle_unpatchify2x2.restype = None
    lib.oracle_max_threads.argtypes = [ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_head_two_pass.argtypes = [f32p, f32p, f32p, f32p, f32p] + [ctypes.c_int] * 7
    lib.oracle_head_two_pass.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def threads_used(threads: int = 0) -> int:
    """Threads the oracle's parallel loops run with for a given ``threads`` argument."""
    return int(_load().oracle_max_threads(int(threads)))


def conv2d(x, w, b=None, stride: int = 1, act: str = "none", layout: str = "NCHW",
           threads: int = 0) -> np.ndarray:
    """2D pad-1 3x3 convolution in fp32; returns fp32 (unrounded) in ``layout``.

    x: [N,C_in,H,W] (NCHW) or [N,H,W,C_in] (NHWC); w: [C_out,C_in,3,3]; b: [C_out] or None.
    """
    x = np.asarray(x)
    if layout == "NHWC":
        x = x.transpose(0, 3, 1, 2)
    elif layout != "NCHW":
        raise ValueError(layout)
    x = _f32(x)
    w = _f32(w)
    N, C_in, H, W = x.shape
    C_out = w.shape[0]
    if w.shape != (C_out, C_in, 3, 3):
        raise ValueError(f"weight shape {w.shape}")
    bb = None if b is None else _f32(b)
    H_out, W_out = (H - 1) // stride + 1, (W - 1) // stride + 1
    y = np.empty((N, C_out, H_out, W_out), np.float32)
    rc = _load().oracle_conv2d(_ptr(x), _ptr(w), _ptr(bb), _ptr(y), N, C_in, C_out, H, W,
                               stride, ACT[act], int(threads))
    if rc != 0:
        raise ValueError("oracle_conv2d: bad arguments")
    return y.transpose(0, 2, 3, 1).copy() if layout == "NHWC" else y


def conv3d_causal(x, w, b=None, carry=None, act: str = "none", layout: str = "NCDHW",
                  threads: int = 0) -> np.ndarray:
    """Causal 3x3x3 convolution in fp32 over [carry(2 frames), x(D frames)].

    x: [N,C_in,D,H,W] (NCDHW) or [N,D,H,W,C_in] (NDHWC); carry: same layout with 2 frames, or
    None for zero frames; w: [C_out,C_in,3,3,3]. Returns fp32 [N,C_out,D,H,W] in ``layout``.
    """
    x = np.asarray(x)
    if layout == "NDHWC":
        x = x.transpose(0, 4, 1, 2, 3)
        if carry is not None:
            carry = np.asarray(carry).transpose(0, 4, 1, 2, 3)
    elif layout != "NCDHW":
        raise ValueError(layout)
    x = _f32(x)
    w = _f32(w)
    N, C_in, D, H, W = x.shape
    C_out = w.shape[0]
    if w.shape != (C_out, C_in, 3, 3, 3):
        raise ValueError(f"weight shape {w.shape}")
    cc = None if carry is None else _f32(carry)
    if cc is not None and cc.shape != (N, C_in, 2, H, W):
        raise ValueError(f"carry shape {cc.shape}")
    bb = None if b is None else _f32(b)
    y = np.empty((N, C_out, D, H, W), np.float32)
    rc = _load().oracle_conv3d_causal(_ptr(x), _ptr(cc), _ptr(w), _ptr(bb), _ptr(y), N, C_in,
                                      C_out, D, H, W, ACT[act], int(threads))
    if rc != 0:
        raise ValueError("oracle_conv3d_causal: bad arguments")
    return y.transpose(0, 2, 3, 4, 1).copy() if layout == "NDHWC" else y


def head_two_pass(x, w, b=None, carry=None, round_g: bool = True, layout: str = "NCDHW", threads: int = 0):
    """The conv_out head (256->12 causal 3x3x3, clamp) computed as the head.cu page's two passes:
    a temporal-only convolution into a 108-channel plane g (rounded to bf16 when round_g), then the
    nine spatial taps summed in fp32 from g plus the bias, then the clamp. Returns fp32 (unrounded)
    [N,12,D,H,W] in ``layout`` (the caller rounds once to the storage type)."""
    x = np.asarray(x)
    if layout == "NDHWC":
        x = x.transpose(0, 4, 1, 2, 3)
        if carry is not None:
            carry = np.asarray(carry).transpose(0, 4, 1, 2, 3)
    x = _f32(x)
    w = _f32(w)
    N, C_in, D, H, W = x.shape
    if w.shape != (12, C_in, 3, 3, 3):
        raise ValueError(f"weight shape {w.shape}")
    cc = None if carry is None else _f32(carry)
    bb = None if b is None else _f32(b)
    y = np.empty((N, 12, D, H, W), np.float32)
    rc = _load().oracle_head_two_pass(_ptr(x), _ptr(cc), _ptr(w), _ptr(bb), _ptr(y), N, C_in, D, H, W,
                                      int(bool(round_g)), int(threads))
    if rc != 0:
        raise ValueError("oracle_head_two_pass: bad arguments")
    return y.transpose(0, 2, 3, 4, 1).copy() if layout == "NDHWC" else y


def round_to(y, dtype: str):
    """Round fp32 values to f16/bf16 (IEEE roundTiesToEven); returns (values as f32, raw bits)."""
    y = _f32(y)
    out = np.empty_like(y)
    bits = np.empty(y.shape, np.uint16)
    _load().oracle_round_to(_ptr(y), _ptr(out), y.size, DTYPE[dtype],
                            bits.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out, bits


def decode_bits(bits, dtype: str) -> np.ndarray:
    """f16/bf16 raw bits -> f32 values, by the oracle's own decoder."""
    lib = _load()
    fn = lib.oracle_f16_to_f32 if dtype == "f16" else lib.oracle_bf16_to_f32
    flat = np.asarray(bits, np.uint16).ravel()
    return np.array([fn(int(v)) for v in flat], np.float32).reshape(np.shape(bits))


def unpatchify2x2(y12) -> np.ndarray:
    """[N,12,D,H,W] -> [N,3,D,2H,2W] with c12 = rgb*4 + dy*2 + dx."""
    y12 = _f32(y12)
    N, C, D, H, W = y12.shape
    if C != 12:
        raise ValueError("unpatchify2x2 needs 12 channels")
    rgb = np.empty((N, 3, D, 2 * H, 2 * W), np.float32)
    _load().oracle_unpatchify2x2(_ptr(y12), _ptr(rgb), N, D, H, W)
    return rgb


def conv2d_chain(x, layers, threads: int = 0) -> np.ndarray:
    """A chain of 2D convs kept in fp32 between layers (no intermediate rounding).

    ``layers`` is a list of dicts with keys w, b, stride, act. x is NCHW.
    """
    y = _f32(x)
    for L in layers:
        y = conv2d(y, L["w"], L.get("b"), stride=L.get("stride", 1), act=L.get("act", "none"),
                   threads=threads)
    return y


def conv3d_chain(x, layers, carries=None, threads: int = 0, layout: str = "NCDHW"):
    """A chain of causal 3D convs in fp32. Returns (y, new_carries).

    Layer i consumes the previous layer's output; its carry is ``carries[i]`` (None = zeros) and
    its new carry is the last two frames of [carry, input] it saw, i.e. of its own input sequence.
    """
    y = _f32(x)
    tdim = 2 if layout == "NCDHW" else 1
    new_carries = []
    for i, L in enumerate(layers):
        c = None if carries is None else carries[i]
        seq = y if c is None else np.concatenate([_f32(c), y], axis=tdim)
        if seq.shape[tdim] >= 2:
            new_carries.append(np.take(seq, [seq.shape[tdim] - 2, seq.shape[tdim] - 1], axis=tdim))
        else:
            zeros = np.zeros_like(np.take(y, [0], axis=tdim))
            new_carries.append(np.concatenate([zeros, y], axis=tdim))
        y = conv3d_causal(y, L["w"], L.get("b"), carry=c, act=L.get("act", "none"), layout=layout,
                          threads=threads)
    return y, new_carries
