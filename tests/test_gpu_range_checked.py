"""The range-checked build (-DDCN_DEBUG_BOUNDS) on the small and ragged cases.

In that build every data-dependent access (bilinear corners from the input
or from a staged window, grad_input reductions, counting-sort cells and
list entries in shared memory, offset/mask/gradient rows, the feature step's
staging copies and stores) checks its bytes against the tensor or buffer it
belongs to; a failed check skips the access and sets a device status word,
and the call returns DCN_ERR_INTERNAL after a synchronisation.  Here every
call must come back DCN_OK (no check failed) with results equal to the
oracle's and the canary guards around the outputs intact.  The status-word
plumbing itself is tested by setting a word from the host.
"""
import ctypes

import pytest
import torch

import test_gpu_parity as P
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300 import build
from deformable_convolution_03_b300.inputs import WORKLOADS, make_dwconv_inputs, make_inputs
from oracle import dwconv as odw
from parity import Guarded, assert_close, check_bwd, check_fwd, f64

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native", "oracle_lib")]


@pytest.fixture(scope="module", autouse=True)
def checked(native):
    path = build.build(debug_bounds=True)
    with B.using_library(path) as L:
        L.dcn_internal_debug_bounds.restype = ctypes.c_int
        L.dcn_internal_bounds_status.restype = ctypes.c_uint
        L.dcn_internal_set_bounds_status.argtypes = [ctypes.c_uint]
        assert L.dcn_internal_debug_bounds() == 1
        yield L


def _status(L):
    return L.dcn_internal_bounds_status()


CASES = P.GEOMS + P.SPLIT + [w for w in P.RAGGED if w.gc in (3, 16, 32)]
FWD = {"tma": {}, "wide": {"fwd_tma": 0}, "general": {"fwd_wide": 0}}
BWD = {"default": {}, "split_halo1": {"bwd_split": 1, "bwd_halo": 1},
       "single_pass": {"bwd_split": 0}}


@pytest.mark.parametrize("mode", sorted(FWD))
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_checked(checked, w, mode, opts):
    opts.update(FWD[mode])
    check_fwd(w, make_inputs(w))
    assert _status(checked) == 0


@pytest.mark.parametrize("mode", sorted(BWD))
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_checked(checked, w, mode, opts):
    opts.update(BWD[mode])
    check_bwd(w, make_inputs(w))
    assert _status(checked) == 0


@pytest.mark.parametrize("fused", [1, 0])
@pytest.mark.parametrize("w", [P.small("cfs_chk_f16", "f16", gc=16, G=4, N=2, H=13, W=11,
                                       offset_std=3.0),
                               P.small("cfs_chk_bf16", "bf16", gc=32, G=2, N=2, H=9, W=14,
                                       softmax=1, remove_center=1, kernel_h=3, kernel_w=3)],
                         ids=lambda w: w.name)
def test_forward_with_centre_feature_scale_checked(checked, w, fused, opts):
    # the gate in the forward's epilogue (x_proj from the staged window) and
    # the two-launch path, against the oracle's composition
    import test_gpu_fused_cfs as F
    opts.set("fwd_cfs", fused)
    t = make_inputs(w)
    logits = F._logits(w)
    assert_close(F._run(w, t, logits), F._expect(w, t, logits), w.dtype, w.name)
    assert _status(checked) == 0


@pytest.mark.parametrize("name", ["t_stage1_f16", "g_stage1_bf16", "fb28_s2d2_f32"])
def test_stage_geometry_checked(checked, name):
    # two images at a configuration's plane size, channels and groups: the
    # production tile and window geometry
    w = WORKLOADS[name].with_(N=2, backward=True)
    t = make_inputs(w, grad=True)
    check_fwd(w, t)
    check_bwd(w, t)
    assert _status(checked) == 0


@pytest.mark.parametrize("dt,C,k", [("f16", 64, 5), ("bf16", 512, 5), ("f32", 128, 3),
                                    ("bf16", 80, 3), ("f32", 64, 7)])
def test_feature_step_checked(checked, dt, C, k):
    t = make_dwconv_inputs(3, 9, 13, C, k, dt, seed=C + k)
    x = t["x"].cuda()
    y = Guarded(tuple(x.shape), x.dtype)
    B.dcn_dwconv_ln_gelu(x, t["weight"].cuda(), t["bias"].cuda(), t["gamma"].cuda(),
                         t["beta"].cuda(), y.t, 1e-6)
    torch.cuda.synchronize()
    y.check("feature step")
    ref = odw.dwconv_ln_gelu(f64(t["x"]), f64(t["weight"]), f64(t["bias"]), f64(t["gamma"]),
                             f64(t["beta"]), 1e-6)
    assert_close(y.t, ref, dt, "feature step (checked build)")
    assert _status(checked) == 0


@pytest.mark.parametrize("ws", [1, 0])
@pytest.mark.parametrize("name,N,K", [("t_stage1_f16", 1, 64), ("g_stage1_bf16", 1, 256)])
def test_forward_with_projection_checked(checked, name, N, K, ws, opts):
    # the forward with its projection in one launch (persistent or per-tile)
    import test_gpu_fused_proj as FP
    opts.update({"fwd_proj": 2, "fwd_proj_ws": ws})
    w = WORKLOADS[name].with_(N=N)
    FP._check(w, K, 32)
    assert _status(checked) == 0


def test_status_word_reports_internal_error(checked):
    # a word set from the host: the next call collects it, reports
    # DCN_ERR_INTERNAL and clears it; the call after that is clean
    w = P.small("plumb", "f32")
    t = make_inputs(w)
    assert checked.dcn_internal_set_bounds_status(5) == B.DCN_OK
    with pytest.raises(B.DCNError) as e:
        check_fwd(w, t)
    assert e.value.status == B.DCN_ERR_INTERNAL
    assert _status(checked) == 5
    check_fwd(w, t)
    assert _status(checked) == 0
