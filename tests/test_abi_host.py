"""The C ABI on the host: symbols, output geometry and every argument check.

Nothing here launches a kernel.  Calls that would pass validation are made
only with the host-side fault hook set (which reports DCN_ERR_CUDA before any
CUDA call), and only where no GPU is present, so no fake pointer can ever
reach a device.
"""
import ctypes
import os
import re

import pytest
import torch

from deformable_convolution_03_b300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# aligned fake device addresses; never dereferenced (every call that uses them
# fails validation, or stops at the fault hook before any CUDA call)
A = 1 << 20

# Tests that hand the library fake device addresses run only where no GPU
# exists: should a check ever regress and let such a call through, it then
# fails at the launch instead of touching a shared device's memory.
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake pointers only where no GPU exists")


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dcn_core.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dcn_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(native):
    names = declared_functions()
    assert set(names) == set(native.EXPORTS), names
    lib = native.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert native.dcn_version() >= 100


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_out_shape_matches_workload_table(native, name):
    w = WORKLOADS[name]
    p = native.Params(dtype=native.DCN_F32, **w.params())
    assert native.dcn_out_shape(p) == (w.H_out, w.W_out)
    assert native.dcn_num_points(p) == w.P
    assert native.dcn_core_bwd_workspace(p) == 0
    p.dtype = native.DCN_BF16
    assert native.dcn_core_bwd_workspace(p) == w.N * w.H * w.W * w.C * 4


@pytest.mark.parametrize("geom", [
    dict(kernel_h=1, kernel_w=1, pad_h=0, pad_w=0),
    dict(kernel_h=5, kernel_w=3, pad_h=2, pad_w=0, stride_w=2),
    dict(kernel_h=3, kernel_w=3, pad_h=0, pad_w=3, dilation_w=3),
    dict(kernel_h=7, kernel_w=7, pad_h=3, pad_w=3, remove_center=1),
    dict(stride_h=3, stride_w=2, dilation_h=2, pad_h=0),
])
def test_out_shape_matches_oracle(native, oracle_lib, geom):
    for H, W in ((7, 6), (16, 9), (31, 31)):
        p = native.Params(N=2, H=H, W=W, G=2, gc=4, **geom)
        q = oracle_lib.Params(N=2, H=H, W=W, G=2, gc=4, **geom)
        assert native.dcn_out_shape(p) == oracle_lib.out_shape(q)
        assert native.dcn_num_points(p) == oracle_lib.num_points(q)


BAD = [
    (dict(dtype=3), "DCN_ERR_DTYPE"),
    (dict(dtype=-1), "DCN_ERR_DTYPE"),
    (dict(N=-1), "DCN_ERR_SHAPE"),
    (dict(H=0), "DCN_ERR_SHAPE"),
    (dict(W=0), "DCN_ERR_SHAPE"),
    (dict(G=0), "DCN_ERR_SHAPE"),
    (dict(gc=0), "DCN_ERR_SHAPE"),
    (dict(kernel_h=0), "DCN_ERR_SHAPE"),
    (dict(stride_w=0), "DCN_ERR_SHAPE"),
    (dict(dilation_h=0), "DCN_ERR_SHAPE"),
    (dict(pad_w=-1), "DCN_ERR_SHAPE"),
    (dict(kernel_h=4, remove_center=1), "DCN_ERR_SHAPE"),
    (dict(softmax=2), "DCN_ERR_SHAPE"),
    (dict(offset_scale=float("nan")), "DCN_ERR_SHAPE"),
    (dict(H=2, pad_h=0), "DCN_ERR_SHAPE"),                  # kernel larger than the image
    (dict(kernel_h=9, kernel_w=9), "DCN_ERR_UNSUPPORTED"),   # 81 points
    (dict(G=1024, gc=128), "DCN_ERR_UNSUPPORTED"),          # 131072 channels
    (dict(H=1 << 23), "DCN_ERR_UNSUPPORTED"),
]


@host_only
@pytest.mark.parametrize("bad,code", BAD)
def test_invalid_parameters_rejected_by_every_entry(native, bad, code):
    p = native.Params(**{**dict(N=1, H=8, W=8, G=2, gc=4), **bad})
    want = getattr(native, code)
    lib = native.lib()
    ho, wo = ctypes.c_int(), ctypes.c_int()
    assert lib.dcn_out_shape(ctypes.byref(p.c()), ctypes.byref(ho), ctypes.byref(wo)) == want
    assert lib.dcn_num_points(ctypes.byref(p.c())) == -want
    assert lib.dcn_core_fwd(ctypes.byref(p.c()), A, A, A, A, None) == want
    assert lib.dcn_core_bwd(ctypes.byref(p.c()), A, A, A, A, A, A, A, A, 1 << 30, None) == want
    assert lib.dcn_core_bwd_workspace(ctypes.byref(p.c())) == 0
    assert code in native.dcn_status_str(want)


@host_only
def test_null_arguments(native):
    lib = native.lib()
    p = native.Params(N=1, H=8, W=8, G=2, gc=4)
    assert lib.dcn_out_shape(None, None, None) == native.DCN_ERR_NULL
    assert lib.dcn_out_shape(ctypes.byref(p.c()), None, None) == native.DCN_ERR_NULL
    assert lib.dcn_core_fwd(None, A, A, A, A, None) == native.DCN_ERR_NULL
    for i in range(4):
        ptrs = [A] * 4
        ptrs[i] = None
        assert lib.dcn_core_fwd(ctypes.byref(p.c()), *ptrs, None) == native.DCN_ERR_NULL
    for i in range(7):
        ptrs = [A] * 7
        ptrs[i] = None
        assert lib.dcn_core_bwd(ctypes.byref(p.c()), *ptrs, None, 0, None) == native.DCN_ERR_NULL


@host_only
def test_fused_forward_argument_errors(native):
    # dcn_core_fwd_cfs / dcn_core_fwd_out: every check that precedes the first
    # CUDA call
    lib = native.lib()
    p = native.Params(N=1, H=8, W=8, G=4, gc=16, dtype=native.DCN_F16)
    pp = ctypes.byref(p.c())
    cfs, out = lib.dcn_core_fwd_cfs, lib.dcn_core_fwd_out
    assert cfs(None, A, A, A, A, A, None) == native.DCN_ERR_NULL
    assert cfs(pp, A, A, A, None, A, None) == native.DCN_ERR_NULL  # the logits
    assert cfs(pp, A, A, A, A + 1, A, None) == native.DCN_ERR_ALIGN
    s2 = native.Params(N=1, H=8, W=8, G=4, gc=16, dtype=native.DCN_F16, stride_h=2, stride_w=2)
    assert cfs(ctypes.byref(s2.c()), A, A, A, A, A, None) == native.DCN_ERR_SHAPE
    assert out(None, A, A, A, None, A, None, 64, A, None, None) == native.DCN_ERR_NULL
    assert out(pp, A, A, A, None, A, None, 0, A, None, None) == native.DCN_ERR_SHAPE
    assert out(pp, A, A, A, None, None, None, 64, A, None, None) == native.DCN_ERR_NULL
    assert out(pp, A, A, A, None, A, None, 64, None, None, None) == native.DCN_ERR_NULL
    assert out(pp, A, A, A, None, A + 1, None, 64, A, None, None) == native.DCN_ERR_ALIGN
    assert out(pp, A, A, A, None, A, A + 1, 64, A, None, None) == native.DCN_ERR_ALIGN
    assert out(ctypes.byref(s2.c()), A, A, A, A, A, None, 64, A, None, None) == native.DCN_ERR_SHAPE
    # no units: nothing to do, nothing touched
    e = native.Params(N=0, H=8, W=8, G=4, gc=16, dtype=native.DCN_F16)
    assert out(ctypes.byref(e.c()), None, None, None, None, A, None, 64, None, None,
               None) == native.DCN_OK


@host_only
def test_misaligned_pointers(native):
    lib = native.lib()
    for dtype, es in ((native.DCN_F32, 4), (native.DCN_F16, 2), (native.DCN_BF16, 2)):
        p = native.Params(N=1, H=8, W=8, G=2, gc=4, dtype=dtype)
        for i in range(4):
            ptrs = [A] * 4
            ptrs[i] = A + (es if i == 1 else 1)  # offset pairs need 2*elem alignment
            assert lib.dcn_core_fwd(ctypes.byref(p.c()), *ptrs, None) == native.DCN_ERR_ALIGN
        for i in range(7):
            ptrs = [A] * 7
            ptrs[i] = A + (es if i == 2 else 1)
            assert lib.dcn_core_bwd(ctypes.byref(p.c()), *ptrs, A, 1 << 30,
                                    None) == native.DCN_ERR_ALIGN
        if dtype != native.DCN_F32:
            assert lib.dcn_core_bwd(ctypes.byref(p.c()), *([A] * 7), A + 8, 1 << 30,
                                    None) == native.DCN_ERR_ALIGN


@host_only
def test_workspace_checks(native):
    lib = native.lib()
    p = native.Params(N=2, H=8, W=8, G=2, gc=4, dtype=native.DCN_F16)
    need = native.dcn_core_bwd_workspace(p)
    assert need == 2 * 8 * 8 * 8 * 4
    assert lib.dcn_core_bwd(ctypes.byref(p.c()), *([A] * 7), None, need,
                            None) == native.DCN_ERR_WORKSPACE
    assert lib.dcn_core_bwd(ctypes.byref(p.c()), *([A] * 7), A, need - 4,
                            None) == native.DCN_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(native):
    lib = native.lib()
    p = native.Params(N=0, H=8, W=8, G=2, gc=4)
    assert lib.dcn_core_fwd(ctypes.byref(p.c()), None, None, None, None, None) == native.DCN_OK
    assert lib.dcn_core_bwd(ctypes.byref(p.c()), *([None] * 8), 0, None) == native.DCN_OK


@host_only
def test_fault_hook_reports_cuda_error(native, opts):
    lib = native.lib()
    p = native.Params(N=1, H=8, W=8, G=2, gc=4, dtype=native.DCN_F16)
    opts.set("fault_inject", 1)
    assert lib.dcn_core_fwd(ctypes.byref(p.c()), A, A, A, A, None) == native.DCN_ERR_CUDA
    assert lib.dcn_core_bwd(ctypes.byref(p.c()), *([A] * 8), 1 << 30, None) == native.DCN_ERR_CUDA
    with pytest.raises(native.DCNError, match="DCN_ERR_CUDA"):
        native.dcn_core_fwd(p, A, A, A, A, stream=0)


def test_status_strings(native):
    for code in range(9):
        assert native.dcn_status_str(code).startswith("DCN_")
    assert "unknown" in native.dcn_status_str(99)


@host_only
def test_merged_layout_argument_checks(native):
    lib = native.lib()
    p = native.Params(N=1, H=8, W=8, G=2, gc=4, dtype=native.DCN_F16)   # P = 9
    for stride in (26, 27, 0, -4):   # below 3P, odd, non-positive
        assert lib.dcn_core_fwd_om(ctypes.byref(p.c()), A, A, stride, A, None) == native.DCN_ERR_SHAPE
        assert lib.dcn_core_bwd_om(ctypes.byref(p.c()), A, A, A, stride, A, A, A, 1 << 30,
                                   None) == native.DCN_ERR_SHAPE
    assert lib.dcn_core_fwd_om(ctypes.byref(p.c()), A, None, 32, A, None) == native.DCN_ERR_NULL
    assert lib.dcn_core_fwd_om(None, A, A, 32, A, None) == native.DCN_ERR_NULL
    assert lib.dcn_core_fwd_om(ctypes.byref(p.c()), A, A + 2, 32, A, None) == native.DCN_ERR_ALIGN
    assert lib.dcn_core_bwd_om(ctypes.byref(p.c()), A, A, A, 32, A, None, A, 1 << 30,
                               None) == native.DCN_ERR_NULL
    bad = native.Params(N=1, H=8, W=8, G=2, gc=4, dtype=7)
    assert lib.dcn_core_fwd_om(ctypes.byref(bad.c()), A, A, 32, A, None) == native.DCN_ERR_DTYPE


# ---- dcn_linear: argument errors are returned before any CUDA call ----------

def _lin(native, M, K, N, dtype=None):
    return native.dcn_linear_params_t(M, K, N, native.DCN_F16 if dtype is None else dtype)


@host_only
def test_linear_argument_errors(native):
    import ctypes
    L = native.lib()
    good = 0x10000  # any 16-byte aligned address; nothing is dereferenced on error
    assert L.dcn_linear(None, good, good, None, good, None) == native.DCN_ERR_NULL
    assert L.dcn_linear(ctypes.byref(_lin(native, 4, 64, 16, 7)), good, good, None, good,
                        None) == native.DCN_ERR_DTYPE
    for M, K, N in ((-1, 64, 16), (4, 0, 16), (4, 64, 0)):
        assert L.dcn_linear(ctypes.byref(_lin(native, M, K, N)), good, good, None, good,
                            None) == native.DCN_ERR_SHAPE
    assert L.dcn_linear(ctypes.byref(_lin(native, 4, 64, 16)), None, good, None, good,
                        None) == native.DCN_ERR_NULL
    assert L.dcn_linear(ctypes.byref(_lin(native, 4, 64, 16)), good + 1, good, None, good,
                        None) == native.DCN_ERR_ALIGN
    assert L.dcn_linear(ctypes.byref(_lin(native, 4, 64, 16)), good, good, good + 1, good,
                        None) == native.DCN_ERR_ALIGN
    # no rows: nothing to do, and nothing is touched
    assert L.dcn_linear(ctypes.byref(_lin(native, 0, 64, 16)), None, None, None, None, None) == native.DCN_OK


# ---- the centre feature scale: argument errors before any CUDA call ----------

def _cfs(native, M, C, G, dtype=None):
    return native.dcn_cfs_params_t(M, C, G, native.DCN_F16 if dtype is None else dtype)


@host_only
def test_centre_feature_scale_argument_errors(native):
    import ctypes
    L = native.lib()
    good = 0x10000
    f, b = L.dcn_center_feature_scale, L.dcn_center_feature_scale_bwd
    assert f(None, good, good, good, good, None) == native.DCN_ERR_NULL
    assert b(None, *([good] * 7), None) == native.DCN_ERR_NULL
    assert f(ctypes.byref(_cfs(native, 4, 64, 4, 9)), good, good, good, good,
             None) == native.DCN_ERR_DTYPE
    for M, C, G in ((-1, 64, 4), (4, 0, 4), (4, 64, 0), (4, 64, 5)):
        p = ctypes.byref(_cfs(native, M, C, G))
        assert f(p, good, good, good, good, None) == native.DCN_ERR_SHAPE
        assert b(p, *([good] * 7), None) == native.DCN_ERR_SHAPE
    assert f(ctypes.byref(_cfs(native, 1 << 34, 64, 4)), good, good, good, good,
             None) == native.DCN_ERR_UNSUPPORTED
    p = ctypes.byref(_cfs(native, 4, 64, 4))
    assert f(p, good, None, good, good, None) == native.DCN_ERR_NULL
    assert b(p, good, good, good, good, good, None, good, None) == native.DCN_ERR_NULL
    assert f(p, good, good + 1, good, good, None) == native.DCN_ERR_ALIGN
    assert b(p, good, good, good, good, good, good, good + 1, None) == native.DCN_ERR_ALIGN
    # no rows: nothing to do, and nothing is touched
    p0 = ctypes.byref(_cfs(native, 0, 64, 4))
    assert f(p0, None, None, None, None, None) == native.DCN_OK
    assert b(p0, *([None] * 7), None) == native.DCN_OK


# ---- the offset branch's feature step: argument errors before any CUDA call --

def _dw(native, N, H, W, C, k, eps=1e-6, dtype=None):
    return native.dcn_dwconv_params_t(N, H, W, C, k, eps,
                                      native.DCN_BF16 if dtype is None else dtype)


@host_only
def test_dwconv_argument_errors(native, opts):
    L = native.lib()
    g = 0x10000
    f = L.dcn_dwconv_ln_gelu
    assert f(None, g, g, g, g, g, g, None) == native.DCN_ERR_NULL
    assert f(ctypes.byref(_dw(native, 1, 8, 8, 64, 5, dtype=7)), g, g, g, g, g, g,
             None) == native.DCN_ERR_DTYPE
    for N, H, W, C, k, eps in ((-1, 8, 8, 64, 5, 1e-6), (1, 0, 8, 64, 5, 1e-6),
                               (1, 8, 0, 64, 5, 1e-6), (1, 8, 8, 0, 5, 1e-6),
                               (1, 8, 8, 64, 4, 1e-6), (1, 8, 8, 64, 0, 1e-6),
                               (1, 8, 8, 64, native.DCN_DW_MAX_KERNEL + 2, 1e-6),
                               (1, 8, 8, 64, 5, -1e-6), (1, 8, 8, 64, 5, float("nan")),
                               (1, 8, 8, 64, 5, float("inf"))):
        assert f(ctypes.byref(_dw(native, N, H, W, C, k, eps)), g, g, g, g, g, g,
                 None) == native.DCN_ERR_SHAPE, (N, H, W, C, k, eps)
    assert f(ctypes.byref(_dw(native, 1, 8, 8, native.DCN_DW_MAX_CHANNELS + 64, 5)), g, g, g, g,
             g, g, None) == native.DCN_ERR_UNSUPPORTED
    assert f(ctypes.byref(_dw(native, 1 << 20, 1 << 10, 1 << 10, 64, 5)), g, g, g, g, g, g,
             None) == native.DCN_ERR_UNSUPPORTED
    p = ctypes.byref(_dw(native, 2, 8, 8, 64, 5))
    for i in (0, 1, 3, 4, 5):  # x, weight, gamma, beta, y; the bias may be NULL
        args = [g] * 6
        args[i] = None
        assert f(p, *args, None) == native.DCN_ERR_NULL, i
        args[i] = g + 1
        assert f(p, *args, None) == native.DCN_ERR_ALIGN, i
    assert f(p, g, g, g + 1, g, g, g, None) == native.DCN_ERR_ALIGN
    # no images: nothing to do, and nothing is touched
    p0 = ctypes.byref(_dw(native, 0, 8, 8, 64, 5))
    assert f(p0, None, None, None, None, None, None, None) == native.DCN_OK
    # a valid call stops at the fault hook, before any CUDA call
    opts.set("fault_inject", 1)
    assert f(p, g, g, None, g, g, g, None) == native.DCN_ERR_CUDA


# ---- the range-checked build ---------------------------------------------------

def test_range_checked_build_exports_every_declared_symbol(native, request):
    from deformable_convolution_03_b300 import build
    path = build.build(debug_bounds=True)
    with native.using_library(path) as L:
        for n in declared_functions():
            assert hasattr(L, n), n
        L.dcn_internal_debug_bounds.restype = ctypes.c_int
        assert L.dcn_internal_debug_bounds() == 1
    # the session's library: the normal one, or the range-checked one when the
    # whole suite runs on it (--range-checked)
    L = native.lib()
    L.dcn_internal_debug_bounds.restype = ctypes.c_int
    assert L.dcn_internal_debug_bounds() == (1 if request.config.getoption("--range-checked") else 0)
