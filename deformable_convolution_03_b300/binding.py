"""ctypes binding of libdcn_b300.so (include/dcn_core.h).

Argument marshalling only: torch tensors become device pointers, the current
torch stream becomes the cudaStream_t, and a non-zero dcn_status_t becomes a
:class:`DCNError`.  Every step of the computation runs in the CUDA library;
there is no other implementation behind these functions.  If the library has
not been built, the first call raises.

The functions named like the C entry points (``dcn_core_fwd`` ...) take
caller-allocated tensors, exactly like the C ABI.  :func:`core_fwd` and
:func:`core_bwd` allocate their results with torch first and then call those.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass, fields

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdcn_b300.so")
# the range-checked build (tests only)
LIB_DEBUG_PATH = os.path.join(_HERE, "libdcn_b300_debug.so")

DCN_F32, DCN_F16, DCN_BF16 = 0, 1, 2
DCN_OK = 0
DCN_ERR_NULL, DCN_ERR_SHAPE, DCN_ERR_DTYPE, DCN_ERR_ALIGN = 1, 2, 3, 4
DCN_ERR_UNSUPPORTED, DCN_ERR_CUDA, DCN_ERR_INTERNAL, DCN_ERR_WORKSPACE = 5, 6, 7, 8
DCN_MAX_POINTS = 64

TORCH_TO_DCN = {torch.float32: DCN_F32, torch.float16: DCN_F16, torch.bfloat16: DCN_BF16}

# Every symbol include/dcn_core.h declares.
EXPORTS = ("dcn_out_shape", "dcn_num_points", "dcn_core_fwd", "dcn_core_fwd_om", "dcn_core_fwd_cfs",
           "dcn_core_fwd_out",
           "dcn_core_bwd_workspace", "dcn_core_bwd", "dcn_core_bwd_om", "dcn_core_bwd_noalloc",
           "dcn_core_fwd_proj", "dcn_linear", "dcn_center_feature_scale",
           "dcn_center_feature_scale_bwd", "dcn_dwconv_ln_gelu", "dcn_wait_timeouts", "dcn_status_str", "dcn_version")
DCN_NOALLOC_SCRATCH_BYTES = 32 << 20
DCN_DW_MAX_KERNEL = 31
DCN_DW_MAX_CHANNELS = 2048


class DCNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dcn_status_str(status)} (status {status})")


class dcn_params_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "H", "W", "G", "gc", "kernel_h", "kernel_w", "stride_h", "stride_w",
        "pad_h", "pad_w", "dilation_h", "dilation_w")] + [
        ("offset_scale", ctypes.c_float), ("softmax", ctypes.c_int),
        ("remove_center", ctypes.c_int), ("dtype", ctypes.c_int)]


@dataclass
class Params:
    """Python mirror of dcn_params_t."""
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
    dtype: int = DCN_F32

    def c(self) -> dcn_params_t:
        return dcn_params_t(**{f.name: getattr(self, f.name) for f in fields(self)})


_lib = None


def _open(path: str) -> ctypes.CDLL:
    """Load a build of the library and declare its entry points' signatures."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with deformable_convolution_03_b300.build.build()")
    L = ctypes.CDLL(path)
    PP = ctypes.POINTER(dcn_params_t)
    vp, ip = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)
    L.dcn_out_shape.argtypes = [PP, ip, ip]
    L.dcn_num_points.argtypes = [PP]
    L.dcn_core_fwd.argtypes = [PP, vp, vp, vp, vp, vp]
    L.dcn_core_bwd_workspace.argtypes = [PP]
    L.dcn_core_bwd_workspace.restype = ctypes.c_size_t
    L.dcn_core_bwd.argtypes = [PP, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.dcn_core_bwd_noalloc.argtypes = [PP, vp, vp, vp, vp, vp, vp, vp, vp]
    L.dcn_core_fwd_om.argtypes = [PP, vp, vp, ctypes.c_int, vp, vp]
    L.dcn_core_fwd_cfs.argtypes = [PP, vp, vp, vp, vp, vp, vp]
    L.dcn_core_fwd_out.argtypes = [PP, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
    L.dcn_core_bwd_om.argtypes = [PP, vp, vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_size_t, vp]
    L.dcn_core_fwd_proj.argtypes = [PP, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, vp]
    L.dcn_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    L.dcn_linear.argtypes = [ctypes.POINTER(dcn_linear_params_t), vp, vp, vp, vp, vp]
    L.dcn_center_feature_scale.argtypes = [ctypes.POINTER(dcn_cfs_params_t), vp, vp, vp, vp, vp]
    L.dcn_center_feature_scale_bwd.argtypes = [ctypes.POINTER(dcn_cfs_params_t)] + [vp] * 8
    L.dcn_dwconv_ln_gelu.argtypes = [ctypes.POINTER(dcn_dwconv_params_t)] + [vp] * 7
    L.dcn_status_str.argtypes = [ctypes.c_int]
    L.dcn_status_str.restype = ctypes.c_char_p
    return L


def lib() -> ctypes.CDLL:
    """The library every call in this module goes through (loaded on first use)."""
    global _lib
    if _lib is None:
        _lib = _open(LIB_PATH)
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route this module's calls through another build of the library (the
    range-checked one, in tests) for the duration of a with-block."""
    global _lib
    prev = _lib
    _lib = _open(path)
    try:
        yield _lib
    finally:
        _lib = prev


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr() if x.numel() else None
    return int(x)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str) -> None:
    if rc != DCN_OK:
        raise DCNError(rc, where)


def dcn_status_str(status: int) -> str:
    return lib().dcn_status_str(int(status)).decode()


def dcn_version() -> int:
    return int(lib().dcn_version())


class dcn_linear_params_t(ctypes.Structure):
    """Mirror of dcn_linear_params_t (include/dcn_core.h)."""
    _fields_ = [("M", ctypes.c_longlong), ("K", ctypes.c_int), ("N", ctypes.c_int),
                ("dtype", ctypes.c_int)]


def dcn_linear(x, w, bias, y, stream=None) -> None:
    """Raw entry point: y = x w^T + bias over the rows of x (all of one dtype)."""
    M, K = int(x.shape[0]), int(x.shape[1])
    p = dcn_linear_params_t(M, K, int(w.shape[0]), TORCH_TO_DCN[x.dtype])
    _check(lib().dcn_linear(ctypes.byref(p), _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
                            _stream(stream)), "dcn_linear")


def linear(x, w, bias=None):
    """y = x w^T + bias on the GPU, x (..., K) channels-last, w (N, K)."""
    for t in (x, w) + ((bias,) if bias is not None else ()):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError("linear: contiguous CUDA tensors of one dtype expected")
    K = x.shape[-1]
    if w.dim() != 2 or w.shape[1] != K or (bias is not None and bias.shape != (w.shape[0],)):
        raise ValueError(f"linear: shapes {tuple(x.shape)}, {tuple(w.shape)} do not match")
    x2 = x.reshape(-1, K)
    y = torch.empty(x2.shape[0], w.shape[0], dtype=x.dtype, device=x.device)
    dcn_linear(x2, w, bias, y, torch.cuda.current_stream(x.device).cuda_stream)
    return y.reshape(*x.shape[:-1], w.shape[0])


class dcn_cfs_params_t(ctypes.Structure):
    """Mirror of dcn_cfs_params_t (include/dcn_core.h)."""
    _fields_ = [("M", ctypes.c_longlong), ("C", ctypes.c_int), ("G", ctypes.c_int),
                ("dtype", ctypes.c_int)]


def dcn_center_feature_scale(core, x_proj, logits, out, G, stream=None) -> None:
    """Raw entry point: out = core * (1 - s) + x_proj * s, s = sigmoid(logits)
    per (row, group); core, x_proj, out (M, C), logits (M, G)."""
    M, C = int(core.shape[0]), int(core.shape[1])
    p = dcn_cfs_params_t(M, C, int(G), TORCH_TO_DCN[core.dtype])
    _check(lib().dcn_center_feature_scale(ctypes.byref(p), _ptr(core), _ptr(x_proj),
                                          _ptr(logits), _ptr(out), _stream(stream)),
           "dcn_center_feature_scale")


def dcn_center_feature_scale_bwd(grad_out, core, x_proj, logits, grad_core, grad_x_proj,
                                 grad_logits, G, stream=None) -> None:
    """Raw entry point: the three gradients of dcn_center_feature_scale."""
    M, C = int(core.shape[0]), int(core.shape[1])
    p = dcn_cfs_params_t(M, C, int(G), TORCH_TO_DCN[core.dtype])
    _check(lib().dcn_center_feature_scale_bwd(
        ctypes.byref(p), _ptr(grad_out), _ptr(core), _ptr(x_proj), _ptr(logits),
        _ptr(grad_core), _ptr(grad_x_proj), _ptr(grad_logits), _stream(stream)),
        "dcn_center_feature_scale_bwd")


def _cfs_args(tensors, C, G):
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != tensors[0].dtype:
            raise ValueError("center_feature_scale: contiguous CUDA tensors of one dtype expected")
    if C % G:
        raise ValueError(f"center_feature_scale: {C} channels do not split into {G} groups")


def center_feature_scale(core, x_proj, logits):
    """The centre feature scale on the GPU: core, x_proj (..., C) channels-last,
    logits (..., G); returns core * (1 - s) + x_proj * s with s = sigmoid(logits)
    per (pixel, group)."""
    C, G = core.shape[-1], logits.shape[-1]
    _cfs_args((core, x_proj, logits), C, G)
    if x_proj.shape != core.shape or logits.shape[:-1] != core.shape[:-1]:
        raise ValueError("center_feature_scale: shapes do not match")
    out = torch.empty_like(core)
    dcn_center_feature_scale(core.reshape(-1, C), x_proj.reshape(-1, C), logits.reshape(-1, G),
                             out.reshape(-1, C), G, torch.cuda.current_stream(core.device).cuda_stream)
    return out


def center_feature_scale_backward(grad_out, core, x_proj, logits):
    """The gradients (grad_core, grad_x_proj, grad_logits) of center_feature_scale."""
    C, G = core.shape[-1], logits.shape[-1]
    _cfs_args((grad_out, core, x_proj, logits), C, G)
    gc, gx, gl = torch.empty_like(core), torch.empty_like(x_proj), torch.empty_like(logits)
    dcn_center_feature_scale_bwd(grad_out.reshape(-1, C), core.reshape(-1, C),
                                 x_proj.reshape(-1, C), logits.reshape(-1, G), gc.reshape(-1, C),
                                 gx.reshape(-1, C), gl.reshape(-1, G), G,
                                 torch.cuda.current_stream(core.device).cuda_stream)
    return gc, gx, gl


class dcn_dwconv_params_t(ctypes.Structure):
    """Mirror of dcn_dwconv_params_t (include/dcn_core.h)."""
    _fields_ = [("N", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("C", ctypes.c_int), ("k", ctypes.c_int), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int)]


def dcn_dwconv_ln_gelu(x, weight, bias, gamma, beta, y, eps: float, stream=None) -> None:
    """Raw entry point: y = GELU(LayerNorm(depthwise k x k conv of x + bias));
    x, y (N, H, W, C), weight (k, k, C), bias (C) or None, gamma, beta (C)."""
    N, H, W, C = (int(v) for v in x.shape)
    p = dcn_dwconv_params_t(N, H, W, C, int(weight.shape[0]), float(eps), TORCH_TO_DCN[x.dtype])
    _check(lib().dcn_dwconv_ln_gelu(ctypes.byref(p), _ptr(x), _ptr(weight), _ptr(bias),
                                    _ptr(gamma), _ptr(beta), _ptr(y), _stream(stream)),
           "dcn_dwconv_ln_gelu")


def dwconv_ln_gelu(x, weight, bias, gamma, beta, eps: float = 1e-6):
    """The offset branch's feature step on the GPU: x (N, H, W, C) channels-last,
    weight (k, k, C) (a depthwise Conv2d weight (C, 1, k, k) permuted to
    (k, k, C)), bias (C) or None, gamma, beta (C); returns a new (N, H, W, C)."""
    ts = (x, weight, gamma, beta) + ((bias,) if bias is not None else ())
    for t in ts:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError("dwconv_ln_gelu: contiguous CUDA tensors of one dtype expected")
    if x.dim() != 4:
        raise ValueError(f"dwconv_ln_gelu: x must be (N, H, W, C), got {tuple(x.shape)}")
    C, k = x.shape[3], weight.shape[0]
    if weight.shape != (k, k, C) or gamma.shape != (C,) or beta.shape != (C,) or (
            bias is not None and bias.shape != (C,)):
        raise ValueError("dwconv_ln_gelu: parameter shapes do not match the channels")
    y = torch.empty_like(x)
    dcn_dwconv_ln_gelu(x, weight, bias, gamma, beta, y, eps,
                       torch.cuda.current_stream(x.device).cuda_stream)
    return y


def dcn_wait_timeouts() -> int:
    """Blocks whose bounded wait for a tensor copy ran out (current device)."""
    n = ctypes.c_ulonglong(0)
    _check(lib().dcn_wait_timeouts(ctypes.byref(n)), "dcn_wait_timeouts")
    return int(n.value)


def dcn_out_shape(p: Params) -> tuple[int, int]:
    ho, wo = ctypes.c_int(), ctypes.c_int()
    _check(lib().dcn_out_shape(ctypes.byref(p.c()), ctypes.byref(ho), ctypes.byref(wo)),
           "dcn_out_shape")
    return ho.value, wo.value


def dcn_num_points(p: Params) -> int:
    r = lib().dcn_num_points(ctypes.byref(p.c()))
    if r < 0:
        raise DCNError(-r, "dcn_num_points")
    return r


def dcn_core_fwd(p: Params, input, offset, mask, output, stream=None) -> None:
    """Raw entry point: pointers (tensors or ints) in, output written in place."""
    _check(lib().dcn_core_fwd(ctypes.byref(p.c()), _ptr(input), _ptr(offset), _ptr(mask),
                              _ptr(output), _stream(stream)), "dcn_core_fwd")


def dcn_core_fwd_cfs(p: Params, input, offset, mask, logits, output, stream=None) -> None:
    """Raw entry point: the core forward followed by the centre feature scale
    with x_proj = input and logits (N, Ho, Wo, G); output written in place."""
    _check(lib().dcn_core_fwd_cfs(ctypes.byref(p.c()), _ptr(input), _ptr(offset), _ptr(mask),
                                  _ptr(logits), _ptr(output), _stream(stream)),
           "dcn_core_fwd_cfs")


def dcn_core_fwd_out(p: Params, input, offset, mask, logits, weight, bias, y, scratch=None,
                     stream=None) -> None:
    """Raw entry point: the core forward (with the centre feature scale when
    logits is given) followed by the output projection y = out weight^T + bias;
    scratch (N, Ho, Wo, C) is needed only where the single launch does not apply."""
    _check(lib().dcn_core_fwd_out(ctypes.byref(p.c()), _ptr(input), _ptr(offset), _ptr(mask),
                                  _ptr(logits), _ptr(weight), _ptr(bias), int(weight.shape[0]),
                                  _ptr(y), _ptr(scratch), _stream(stream)),
           "dcn_core_fwd_out")


def dcn_core_bwd_workspace(p: Params) -> int:
    return int(lib().dcn_core_bwd_workspace(ctypes.byref(p.c())))


def dcn_core_bwd(p: Params, grad_out, input, offset, mask, grad_input, grad_offset, grad_mask,
                 workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    """Raw entry point: all three gradients written in place."""
    if workspace_bytes is None:
        workspace_bytes = (workspace.numel() * workspace.element_size()
                           if isinstance(workspace, torch.Tensor) else 0)
    _check(lib().dcn_core_bwd(ctypes.byref(p.c()), _ptr(grad_out), _ptr(input), _ptr(offset),
                              _ptr(mask), _ptr(grad_input), _ptr(grad_offset), _ptr(grad_mask),
                              _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "dcn_core_bwd")


def dcn_core_fwd_om(p: Params, input, offset_mask, row_stride: int, output, stream=None) -> None:
    """Forward with DCNv4's merged offset/mask tensor (N, Ho, Wo, G, row_stride)."""
    _check(lib().dcn_core_fwd_om(ctypes.byref(p.c()), _ptr(input), _ptr(offset_mask),
                                 int(row_stride), _ptr(output), _stream(stream)),
           "dcn_core_fwd_om")


def dcn_core_fwd_proj(p: Params, input, feat, weight, bias, row_stride: int, output,
                      offset_mask=None, stream=None) -> None:
    """Raw entry point: the forward with the merged offset/mask projection
    feat (N, Ho, Wo, K) x weight (G*row_stride, K)^T + bias in the same launch;
    the rows are also written to offset_mask (N, Ho, Wo, G, row_stride) when
    given."""
    _check(lib().dcn_core_fwd_proj(ctypes.byref(p.c()), _ptr(input), _ptr(feat),
                                   int(feat.shape[-1]), _ptr(weight), _ptr(bias),
                                   int(row_stride), _ptr(output), _ptr(offset_mask),
                                   _stream(stream)), "dcn_core_fwd_proj")


def dcn_core_bwd_om(p: Params, grad_out, input, offset_mask, row_stride: int, grad_input,
                    grad_offset_mask, workspace=None, workspace_bytes: int | None = None,
                    stream=None) -> None:
    """Backward with the merged layout; grad_offset_mask has offset_mask's layout."""
    if workspace_bytes is None:
        workspace_bytes = (workspace.numel() * workspace.element_size()
                           if isinstance(workspace, torch.Tensor) else 0)
    _check(lib().dcn_core_bwd_om(ctypes.byref(p.c()), _ptr(grad_out), _ptr(input),
                                 _ptr(offset_mask), int(row_stride), _ptr(grad_input),
                                 _ptr(grad_offset_mask), _ptr(workspace), int(workspace_bytes),
                                 _stream(stream)),
           "dcn_core_bwd_om")


def dcn_core_bwd_noalloc(p: Params, grad_out, input, offset, mask, grad_input, grad_offset,
                         grad_mask, stream=None) -> None:
    """The backward without a workspace: for callers that may not allocate
    device memory where they run it.  The float32 accumulator that float16 /
    bfloat16 need comes from the library's own static device array
    (DCN_NOALLOC_SCRATCH_BYTES), shared by all calls on a device, so calls
    must not overlap on the GPU."""
    _check(lib().dcn_core_bwd_noalloc(ctypes.byref(p.c()), _ptr(grad_out), _ptr(input),
                                      _ptr(offset), _ptr(mask), _ptr(grad_input),
                                      _ptr(grad_offset), _ptr(grad_mask), _stream(stream)),
           "dcn_core_bwd_noalloc")


# ---- tensor-level convenience: shapes from the tensors, results allocated ----

def params_for(input: torch.Tensor, G: int, **geom) -> Params:
    """Params for a channels-last input tensor (N, H, W, G*gc) and G groups."""
    if input.dim() != 4:
        raise ValueError("input must be (N, H, W, G*gc)")
    N, H, W, C = input.shape
    if C % G:
        raise ValueError(f"channels {C} not divisible by groups {G}")
    if input.dtype not in TORCH_TO_DCN:
        raise TypeError(f"unsupported dtype {input.dtype}")
    return Params(N=N, H=H, W=W, G=G, gc=C // G, dtype=TORCH_TO_DCN[input.dtype], **geom)


def _expect(t: torch.Tensor, name: str, shape: tuple, dtype, device) -> None:
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def shapes(p: Params) -> dict:
    ho, wo = dcn_out_shape(p)
    P = dcn_num_points(p)
    C = p.G * p.gc
    return {"input": (p.N, p.H, p.W, C), "offset": (p.N, ho, wo, p.G, P, 2),
            "mask": (p.N, ho, wo, p.G, P), "output": (p.N, ho, wo, C)}


def core_fwd(input, offset, mask, G: int, stream=None, out=None, **geom) -> torch.Tensor:
    """output = the core op on CUDA tensors; geom: kernel_h ... remove_center."""
    p = params_for(input, G, **geom)
    sh = shapes(p)
    if input.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for name, t in (("input", input), ("offset", offset), ("mask", mask)):
        _expect(t, name, sh[name], input.dtype, input.device)
    if out is None:
        out = torch.empty(sh["output"], dtype=input.dtype, device=input.device)
    _expect(out, "out", sh["output"], input.dtype, input.device)
    dcn_core_fwd(p, input, offset, mask, out, stream)
    return out


def core_bwd(grad_out, input, offset, mask, G: int, stream=None, **geom):
    """(grad_input, grad_offset, grad_mask) on CUDA tensors."""
    p = params_for(input, G, **geom)
    sh = shapes(p)
    if input.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for name, t in (("input", input), ("offset", offset), ("mask", mask)):
        _expect(t, name, sh[name], input.dtype, input.device)
    _expect(grad_out, "grad_out", sh["output"], input.dtype, input.device)
    gi = torch.empty_like(input)
    go = torch.empty_like(offset)
    gm = torch.empty_like(mask)
    nbytes = dcn_core_bwd_workspace(p)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=input.device) if nbytes else None
    dcn_core_bwd(p, grad_out, input, offset, mask, gi, go, gm, ws, nbytes, stream)
    return gi, go, gm


class DCNCoreFunction(torch.autograd.Function):
    """autograd wrapper: forward and backward both run the CUDA library."""

    @staticmethod
    def forward(ctx, input, offset, mask, G, geom):
        ctx.save_for_backward(input, offset, mask)
        ctx.G, ctx.geom = G, geom
        return core_fwd(input, offset, mask, G, **geom)

    @staticmethod
    def backward(ctx, grad_out):
        input, offset, mask = ctx.saved_tensors
        gi, go, gm = core_bwd(grad_out.contiguous(), input, offset, mask, ctx.G, **ctx.geom)
        return gi, go, gm, None, None


def dcn_core(input, offset, mask, G: int, **geom) -> torch.Tensor:
    """Differentiable core op (DCNv3 with softmax=1, DCNv4 with softmax=0)."""
    return DCNCoreFunction.apply(input, offset, mask, G, geom)
