"""Python binding of libx3conv, the GB300 (sm_103a) 3x3 / causal 3x3x3 convolution library.

The functions below carry the C ABI's names (``include/x3conv.h``) and only marshal arguments:
every step of the computation runs in the library's CUDA kernels. PyTorch provides the device
memory and the stream. The library must have been built (``x3x3_convolution_gb300.build.build()``
or ``__graft_entry__.build()``); without it every call raises ``RuntimeError`` - there is no
CPU fallback.

Convenience wrappers (:class:`Conv`, :class:`ConvStack`) take torch tensors and manage the plan
and the packed weights; they are argument plumbing over the same entry points.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

X3_OK, X3_ERR_INVALID, X3_ERR_UNSUPPORTED, X3_ERR_CUDA, X3_ERR_OOM, X3_ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "X3_OK", 1: "X3_ERR_INVALID", 2: "X3_ERR_UNSUPPORTED", 3: "X3_ERR_CUDA",
                4: "X3_ERR_OOM", 5: "X3_ERR_TIMEOUT"}
LAYOUT = {"NCHW": 0, "NHWC": 1, "NCDHW": 2, "NDHWC": 3}
DTYPE = {"f16": 0, "bf16": 1}
ACT = {"none": 0, "relu": 1, "clamp": 2}
KERNEL = {"auto": 0, "igemm": 1, "direct": 2, "head_two_pass": 3, "head_split": 4, "head_stencil": 5}


class ConvDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "dims", "N", "C_in", "C_out", "D", "H", "W", "stride", "layout", "dtype", "act", "has_bias",
        "unpatchify2x2", "kernel", "band_lo", "band_rows", "H_global")]


class X3Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libx3conv.so (raises RuntimeError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libx3conv.so is not built ({_build.LIB}); run x3x3_convolution_gb300.build.build()")
    lib = ctypes.CDLL(_build.LIB)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "conv_plan_create": ([ctypes.POINTER(ConvDesc), ctypes.POINTER(vp)], i),
        "conv_plan_destroy": ([vp], None),
        "conv_plan_kernel_name": ([vp], ctypes.c_char_p),
        "conv_plan_launches": ([vp], i),
        "conv_plan_describe": ([vp, ctypes.c_char_p, sz], i),
        "conv_packed_weight_bytes": ([vp], sz),
        "conv_pack_weights": ([vp, vp, vp, vp], i),
        "conv_forward": ([vp, vp, vp, vp, vp, vp, vp], i),
        "conv_stack_workspace_bytes": ([pp, i], sz),
        "conv_stack_forward": ([pp, i, vp, pp, i, pp, pp, vp, vp, sz, vp], i),
        "conv_device_status": ([i], i),
        "conv_head_g_bytes": ([vp], sz),
        "conv_head_two_pass": ([vp, vp, vp, vp, vp, vp, vp, vp], i),
        "conv_selftest_wait_timeout": ([i, vp], i),
        "conv_last_error": ([], ctypes.c_char_p),
        "conv_version": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status):
    if status != X3_OK:
        raise X3Error(status, conv_last_error())


def _ptrs(seq):
    arr = (ctypes.c_void_p * len(seq))(*[p if p else None for p in seq])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


# ------------------------------------------------------------------ raw entry points (C ABI names)

def conv_plan_create(desc: ConvDesc) -> int:
    plan = ctypes.c_void_p()
    _check(load().conv_plan_create(ctypes.byref(desc), ctypes.byref(plan)))
    return plan.value


def conv_plan_destroy(plan: int) -> None:
    load().conv_plan_destroy(plan)


def conv_plan_kernel_name(plan: int) -> str:
    return load().conv_plan_kernel_name(plan).decode()


def conv_plan_describe(plan: int) -> dict:
    import json
    n = load().conv_plan_describe(plan, None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    load().conv_plan_describe(plan, buf, n + 1)
    return json.loads(buf.value.decode())


def conv_plan_launches(plan: int) -> int:
    return load().conv_plan_launches(plan)


def conv_packed_weight_bytes(plan: int) -> int:
    return load().conv_packed_weight_bytes(plan)


def conv_pack_weights(plan: int, w: int, w_packed: int, stream: int = 0) -> None:
    _check(load().conv_pack_weights(plan, w, w_packed, stream))


def conv_forward(plan: int, x: int, carry, w_packed: int, bias, y: int, stream: int = 0) -> None:
    _check(load().conv_forward(plan, x, carry or None, w_packed, bias or None, y, stream))


def conv_stack_workspace_bytes(plans) -> int:
    p, _keep = _ptrs(plans)
    return load().conv_stack_workspace_bytes(p, len(plans))


def conv_stack_forward(plans, x: int, carries, carry_valid: int, w_packed, bias, y: int, workspace,
                       workspace_bytes: int, stream: int = 0) -> None:
    p, k1 = _ptrs(plans)
    c, k2 = _ptrs(carries) if carries is not None else (None, None)
    w, k3 = _ptrs(w_packed)
    b, k4 = _ptrs(bias)
    _check(load().conv_stack_forward(p, len(plans), x, c, int(carry_valid), w, b, y, workspace or None,
                                     workspace_bytes, stream))


def conv_head_g_bytes(plan: int) -> int:
    return load().conv_head_g_bytes(plan)


def conv_head_two_pass(plan: int, x: int, carry, w_packed: int, bias, g: int, y: int, stream: int = 0) -> None:
    _check(load().conv_head_two_pass(plan, x, carry or None, w_packed, bias or None, g, y, stream))


def conv_device_status(reset: int = 0) -> int:
    return load().conv_device_status(reset)


def conv_selftest_wait_timeout(limit_ms: int, stream: int = 0) -> None:
    _check(load().conv_selftest_wait_timeout(int(limit_ms), stream))


def conv_last_error() -> str:
    return load().conv_last_error().decode()


def conv_version() -> str:
    return load().conv_version().decode()


# ------------------------------------------------------------------ torch plumbing

def _torch():
    import torch
    return torch


def make_desc(dims, N, C_in, C_out, H, W, D=1, stride=1, layout=None, dtype="bf16", act="none",
              has_bias=True, unpatchify2x2=False, kernel="auto", band_lo=0, band_rows=0, H_global=0) -> ConvDesc:
    """A layer descriptor. band_lo / band_rows / H_global select the banded mode (output rows
    [band_lo, band_lo + band_rows) of an H_global-row image; H = the band's rows plus its existing halo
    rows); all 0 = the whole plane."""
    if layout is None:
        layout = "NDHWC" if dims == 3 else "NCHW"
    return ConvDesc(dims, N, C_in, C_out, D if dims == 3 else 1, H, W, stride, LAYOUT[layout],
                    DTYPE[dtype], ACT[act], int(bool(has_bias)), int(bool(unpatchify2x2)),
                    KERNEL[kernel], int(band_lo), int(band_rows), int(H_global))


def band_input_rows(band_lo, band_rows, H_global):
    """The global input rows [lo, hi) a band of output rows needs (its rows plus the halo rows that
    exist): the H of its descriptor is hi - lo."""
    return max(band_lo - 1, 0), min(band_lo + band_rows + 1, H_global)


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Conv:
    """One convolution layer: a plan plus its packed weights (device memory held by torch)."""

    def __init__(self, desc: ConvDesc, weight, bias=None, device="cuda"):
        torch = _torch()
        self.desc = desc
        self.plan = conv_plan_create(desc)
        self.kernel_name = conv_plan_kernel_name(self.plan)
        nbytes = conv_packed_weight_bytes(self.plan)
        self.w_packed = torch.empty(nbytes // 2 + 128, dtype=torch.int16, device=device)
        off = (-self.w_packed.data_ptr()) % 256
        self._wp = self.w_packed.data_ptr() + off
        w = weight.contiguous()
        conv_pack_weights(self.plan, w.data_ptr(), self._wp, _stream(None))
        self._w_keep = w
        self.bias = None if bias is None else bias.contiguous()
        torch.cuda.current_stream().synchronize()
        self._w_keep = None

    @property
    def H_out(self):
        if self.desc.H_global:
            return self.desc.band_rows
        return (self.desc.H - 1) // self.desc.stride + 1

    @property
    def W_out(self):
        return (self.desc.W - 1) // self.desc.stride + 1

    def out_shape(self):
        d = self.desc
        Ho, Wo = self.H_out, self.W_out
        lay = [k for k, v in LAYOUT.items() if v == d.layout][0]
        if d.unpatchify2x2:
            if lay == "NDHWC":
                return (d.N, d.D, 2 * Ho, 2 * Wo, 3)
            if lay == "NCDHW":
                return (d.N, 3, d.D, 2 * Ho, 2 * Wo)
            if lay == "NHWC":
                return (d.N, 2 * Ho, 2 * Wo, 3)
            return (d.N, 3, 2 * Ho, 2 * Wo)
        return {"NCHW": (d.N, d.C_out, Ho, Wo), "NHWC": (d.N, Ho, Wo, d.C_out),
                "NCDHW": (d.N, d.C_out, d.D, Ho, Wo), "NDHWC": (d.N, d.D, Ho, Wo, d.C_out)}[lay]

    def __call__(self, x, carry=None, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.out_shape(), dtype=x.dtype, device=x.device)
        if self.kernel_name in ("head_two_pass", "head_split"):
            gb = conv_head_g_bytes(self.plan)
            if getattr(self, "_g", None) is None or self._g.numel() * 2 < gb:
                self._g = torch.empty(gb // 2, dtype=torch.int16, device=x.device)
            conv_head_two_pass(self.plan, x.data_ptr(), None if carry is None else carry.data_ptr(), self._wp,
                               None if self.bias is None else self.bias.data_ptr(), self._g.data_ptr(),
                               out.data_ptr(), _stream(stream))
            return out
        conv_forward(self.plan, x.data_ptr(), None if carry is None else carry.data_ptr(), self._wp,
                     None if self.bias is None else self.bias.data_ptr(), out.data_ptr(), _stream(stream))
        return out

    def __del__(self):
        try:
            if getattr(self, "plan", None):
                conv_plan_destroy(self.plan)
                self.plan = None
        except Exception:
            pass


class ConvStack:
    """Chained layers run by conv_stack_forward with a caller-held workspace and per-layer carries."""

    def __init__(self, layers):
        torch = _torch()
        self.layers = list(layers)
        self.plans = [L.plan for L in self.layers]
        ws = conv_stack_workspace_bytes(self.plans)
        self.ws_bytes = ws
        self.workspace = torch.empty(max(ws, 1) + 256, dtype=torch.uint8, device="cuda")
        self._ws = self.workspace.data_ptr() + ((-self.workspace.data_ptr()) % 256)

    def __call__(self, x, carries=None, carry_valid=False, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.layers[-1].out_shape(), dtype=x.dtype, device=x.device)
        cp = None if carries is None else [None if c is None else c.data_ptr() for c in carries]
        conv_stack_forward(self.plans, x.data_ptr(), cp, int(bool(carry_valid)),
                           [L._wp for L in self.layers],
                           [None if L.bias is None else L.bias.data_ptr() for L in self.layers],
                           out.data_ptr(), self._ws if self.ws_bytes else None, self.ws_bytes,
                           _stream(stream))
        return out
