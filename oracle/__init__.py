"""The oracle: a plain binary64 CPU implementation of the DCNv3/DCNv4 core op.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The product (the CUDA library and
its Python binding) never imports, links or calls it, and shares no code with
it.  See ``dcn_oracle.c`` for the passages each step follows.

This module is argument marshalling around ``libdcn_oracle.so`` (built from
``dcn_oracle.c`` by :func:`build`): numpy binary64 arrays in, numpy arrays out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcn_oracle.c")
_LIB = os.path.join(_HERE, "libdcn_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE binary64, no fused contractions)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "H", "W", "G", "gc", "kernel_h", "kernel_w", "stride_h", "stride_w",
        "pad_h", "pad_w", "dilation_h", "dilation_w")] + [
        ("offset_scale", ctypes.c_double),
        ("softmax", ctypes.c_int), ("remove_center", ctypes.c_int), ("coord_f32", ctypes.c_int)]


@dataclass
class Params:
    """Shape and configuration of one core-op call (channels-last tensors)."""
    N: int
    H: int
    W: int
    G: int
    gc: int
    kernel_h: int = 3
    kernel_w: int = 3
    stride_h: int = 1
    stride_w: int = 1
    pad_h: int = 1
    pad_w: int = 1
    dilation_h: int = 1
    dilation_w: int = 1
    offset_scale: float = 1.0
    softmax: int = 0
    remove_center: int = 0
    coord_f32: int = 0

    def _c(self) -> _Params:
        return _Params(**{k: getattr(self, k) for k, _ in _Params._fields_})


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Params)
        D = ctypes.POINTER(ctypes.c_double)
        I = ctypes.POINTER(ctypes.c_int)
        lib.dcno_out_shape.argtypes = [P, I, I]
        lib.dcno_taps.argtypes = [P, I, I]
        lib.dcno_forward.argtypes = [P, D, D, D, D]
        lib.dcno_forward_pixels.argtypes = [P, D, D, D, ctypes.POINTER(ctypes.c_longlong),
                                            ctypes.c_long, D]
        lib.dcno_backward.argtypes = [P, D, D, D, D, D, D, D]
        lib.dcno_backward_pixels.argtypes = [P, D, D, D, D, ctypes.POINTER(ctypes.c_longlong),
                                             ctypes.c_long, D, D, D]
        lib.dcno_set_threads.argtypes = [ctypes.c_int]
        lib.dcno_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def out_shape(p: Params) -> tuple[int, int]:
    ho, wo = ctypes.c_int(), ctypes.c_int()
    if _load().dcno_out_shape(ctypes.byref(p._c()), ctypes.byref(ho), ctypes.byref(wo)) != 0:
        raise ValueError("invalid parameters: %r" % (p,))
    return ho.value, wo.value


def taps(p: Params) -> list[tuple[int, int]]:
    """(tap_x, tap_y) of the P sampling points, in the order of the offset and mask."""
    kk = p.kernel_h * p.kernel_w
    tx, ty = (ctypes.c_int * kk)(), (ctypes.c_int * kk)()
    n = _load().dcno_taps(ctypes.byref(p._c()), tx, ty)
    return [(tx[i], ty[i]) for i in range(n)]


def num_points(p: Params) -> int:
    return p.kernel_h * p.kernel_w - (1 if p.remove_center else 0)


def _check(p: Params, input, offset, mask):
    ho, wo = out_shape(p)
    P = num_points(p)
    C = p.G * p.gc
    input, offset, mask = _f64(input), _f64(offset), _f64(mask)
    if input.size != p.N * p.H * p.W * C:
        raise ValueError("input size")
    if offset.size != p.N * ho * wo * p.G * P * 2:
        raise ValueError("offset size")
    if mask.size != p.N * ho * wo * p.G * P:
        raise ValueError("mask size")
    return ho, wo, P, C, input, offset, mask


def forward(p: Params, input, offset, mask) -> np.ndarray:
    """output (N, Ho, Wo, G*gc) in binary64."""
    ho, wo, P, C, input, offset, mask = _check(p, input, offset, mask)
    out = np.zeros((p.N, ho, wo, C), dtype=np.float64)
    if _load().dcno_forward(ctypes.byref(p._c()), _dp(input), _dp(offset), _dp(mask), _dp(out)):
        raise ValueError("oracle forward rejected the parameters")
    return out


def forward_pixels(p: Params, input, offset, mask, pixels) -> np.ndarray:
    """Forward at flat output pixels n*Ho*Wo + ho*Wo + wo only: (len(pixels), G*gc)."""
    ho, wo, P, C, input, offset, mask = _check(p, input, offset, mask)
    pix = np.ascontiguousarray(np.asarray(pixels, dtype=np.int64))
    out = np.zeros((pix.size, C), dtype=np.float64)
    rc = _load().dcno_forward_pixels(
        ctypes.byref(p._c()), _dp(input), _dp(offset), _dp(mask),
        pix.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)), pix.size, _dp(out))
    if rc:
        raise ValueError("oracle forward_pixels rejected the arguments")
    return out


def backward(p: Params, grad_out, input, offset, mask):
    """(grad_input, grad_offset, grad_mask) of <grad_out, forward(...)>, binary64."""
    ho, wo, P, C, input, offset, mask = _check(p, input, offset, mask)
    grad_out = _f64(grad_out)
    if grad_out.size != p.N * ho * wo * C:
        raise ValueError("grad_out size")
    gi = np.zeros((p.N, p.H, p.W, C), dtype=np.float64)
    go = np.zeros((p.N, ho, wo, p.G, P, 2), dtype=np.float64)
    gm = np.zeros((p.N, ho, wo, p.G, P), dtype=np.float64)
    if _load().dcno_backward(ctypes.byref(p._c()), _dp(grad_out), _dp(input), _dp(offset),
                             _dp(mask), _dp(gi), _dp(go), _dp(gm)):
        raise ValueError("oracle backward rejected the parameters")
    return gi, go, gm


def backward_pixels(p: Params, grad_out, input, offset, mask, pixels):
    """Backward restricted to flat output pixels: (grad_input from their scatter
    only, grad_offset (len, G, P, 2), grad_mask (len, G, P))."""
    ho, wo, P, C, input, offset, mask = _check(p, input, offset, mask)
    grad_out = _f64(grad_out)
    pix = np.ascontiguousarray(np.asarray(pixels, dtype=np.int64))
    gi = np.zeros((p.N, p.H, p.W, C), dtype=np.float64)
    go = np.zeros((pix.size, p.G, P, 2), dtype=np.float64)
    gm = np.zeros((pix.size, p.G, P), dtype=np.float64)
    if _load().dcno_backward_pixels(ctypes.byref(p._c()), _dp(grad_out), _dp(input), _dp(offset),
                                    _dp(mask), pix.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
                                    pix.size, _dp(gi), _dp(go), _dp(gm)):
        raise ValueError("oracle backward_pixels rejected the arguments")
    return gi, go, gm


def set_threads(n: int) -> None:
    _load().dcno_set_threads(int(n))


def max_threads() -> int:
    return int(_load().dcno_max_threads())
