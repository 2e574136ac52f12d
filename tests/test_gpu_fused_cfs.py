"""The core forward with the centre feature scale (dcn_core_fwd_cfs) against
the oracle's composition: the core op (oracle.forward, binary64) and then the
gate with x_proj the core's own input (oracle/proj.py center_feature_scale).

The single launch (16-bit storage, the gate applied to the core's float32 sums
before their one rounding) and the two launches (the core rounded first, then
the gate in place) both meet the oracle within R12's 16-bit tolerance, and
they differ by at most the one extra rounding.  Outputs sit between canary
guards."""
import numpy as np
import pytest
import torch

import oracle
from oracle import proj
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import DTYPES, WORKLOADS, make_inputs
from parity import Guarded, assert_close, f64, lib_params, oracle_params
from test_gpu_parity import small

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native", "oracle_lib")]

ROUND = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}


def _logits(w, seed=5):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(w.N, w.H_out, w.W_out, w.G, generator=g) * 2).to(DTYPES[w.dtype])


def _run(w, t, logits):
    out = Guarded((w.N, w.H_out, w.W_out, w.C), DTYPES[w.dtype])
    B.dcn_core_fwd_cfs(lib_params(w), t["input"].cuda(), t["offset"].cuda(), t["mask"].cuda(),
                       logits.cuda(), out.t)
    torch.cuda.synchronize()
    out.check("output")
    return out.t


def _expect(w, t, logits):
    core = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    M = w.N * w.H_out * w.W_out
    return proj.center_feature_scale(core.reshape(M, w.C), f64(t["input"]).reshape(M, w.C),
                                     f64(logits).reshape(M, w.G), w.G).reshape(core.shape)


def _check(w, opts, seed=5):
    t = make_inputs(w)
    logits = _logits(w, seed)
    ref = _expect(w, t, logits)
    fused = _run(w, t, logits)
    assert_close(fused, ref, w.dtype, f"{w.name} fused")
    opts.set("fwd_cfs", 0)
    two = _run(w, t, logits)
    opts.set("fwd_cfs", 1)
    assert_close(two, ref, w.dtype, f"{w.name} two launches")
    # the two ways differ by the core's rounding to the storage type, scaled by
    # (1 - s), and each result's own rounding
    u = ROUND[w.dtype]
    d = np.abs(f64(fused) - f64(two))
    bound = 3 * u * (np.abs(ref) + np.abs(f64(t["input"])) + 1e-30) + 2 * u * np.abs(ref).max()
    assert np.all(d <= bound), f"{w.name}: single and two launches differ by {d.max()}"
    return fused


# the FlashInternImage-T stages at two images, InternImage-G stage 1 (DCNv3
# softmax, gc 32) with and without its centre tap
STAGES = [("t_stage1_f16", 2), ("t_stage2_bf16", 2), ("t_stage3_bf16", 2), ("t_stage4_bf16", 4),
          ("g_stage1_bf16", 1), ("g_stage1_rc_bf16", 1)]


@pytest.mark.parametrize("name,N", STAGES, ids=[s[0] for s in STAGES])
def test_stage_shapes(name, N, opts):
    _check(WORKLOADS[name].with_(N=N), opts)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("gc,G", [(8, 4), (16, 4), (16, 8), (32, 2)])
@pytest.mark.parametrize("sm,rc", [(0, 0), (1, 0), (1, 1)])
def test_ragged_planes(dt, gc, G, sm, rc, opts):
    # 13 x 11 pixels: ragged tiles both ways; offsets N(0, 3) send some samples
    # past the window (its far path) while x_proj still comes from the window
    w = small(f"cfs_{dt}_{gc}_{G}_{sm}{rc}", dt, gc=gc, G=G, N=2, H=13, W=11, softmax=sm,
              remove_center=rc, offset_std=3.0)
    _check(w, opts, seed=gc + G)


@pytest.mark.parametrize("geom", ["k5", "d2", "k7rc", "k1", "os_half"])
def test_same_size_geometries(geom, opts):
    # every geometry whose output keeps the input's size: 5 x 5 with padding 2,
    # 3 x 3 at dilation 2 with padding 2, 7 x 7 without its centre, 1 x 1, and
    # an offset scale of 1/2
    over = {"k5": dict(kernel_h=5, kernel_w=5, pad_h=2, pad_w=2),
            "d2": dict(dilation_h=2, dilation_w=2, pad_h=2, pad_w=2),
            "k7rc": dict(kernel_h=7, kernel_w=7, pad_h=3, pad_w=3, remove_center=1, softmax=1),
            "k1": dict(kernel_h=1, kernel_w=1, pad_h=0, pad_w=0),
            "os_half": dict(offset_scale=0.5, softmax=1)}[geom]
    w = small(f"cfs_g_{geom}", "bf16", gc=16, G=4, N=2, H=17, W=19, **over)
    _check(w, opts)


def test_float32_two_launches(opts):
    # float32 storage always takes the two launches
    w = small("cfs_f32", "f32", gc=16, G=4, N=2, H=12, W=10)
    t = make_inputs(w)
    logits = _logits(w)
    assert_close(_run(w, t, logits), _expect(w, t, logits), "f32", "f32")


def test_gate_extremes(opts):
    # logits of -60 and +60: the output is the core, or the input, exactly as
    # rounded (the gate is 0 or 1 to float32)
    w = WORKLOADS["t_stage1_f16"].with_(N=1)
    t = make_inputs(w)
    for lv, want in ((-60.0, "core"), (60.0, "input")):
        logits = torch.full((w.N, w.H_out, w.W_out, w.G), lv, dtype=DTYPES[w.dtype])
        out = _run(w, t, logits)
        if want == "input":
            assert torch.equal(out.cpu(), t["input"])
        else:
            core = torch.empty_like(out)
            B.dcn_core_fwd(lib_params(w), t["input"].cuda(), t["offset"].cuda(),
                           t["mask"].cuda(), core)
            torch.cuda.synchronize()
            assert torch.equal(out, core)


def test_shape_and_argument_errors():
    w = small("cfs_err", "f16", gc=16, G=4, N=1, H=9, W=9)
    t = {k: v.cuda() for k, v in make_inputs(w).items()}
    logits = _logits(w).cuda()
    out = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=torch.float16, device="cuda")
    with pytest.raises(B.DCNError) as e:
        B.dcn_core_fwd_cfs(lib_params(w), t["input"], t["offset"], t["mask"], None, out)
    assert e.value.status == B.DCN_ERR_NULL
    # an output smaller than the input (no padding), and a strided one
    for name, over in (("nopad", dict(pad_h=0, pad_w=0)), ("s2", dict(stride_h=2, stride_w=2))):
        v = small(f"cfs_err_{name}", "f16", gc=16, G=4, N=1, H=9, W=9, **over)
        tv = {k: x.cuda() for k, x in make_inputs(v).items()}
        o = torch.empty(v.N, v.H_out, v.W_out, v.C, dtype=torch.float16, device="cuda")
        lg = _logits(v).cuda()
        with pytest.raises(B.DCNError) as e:
            B.dcn_core_fwd_cfs(lib_params(v), tv["input"], tv["offset"], tv["mask"], lg, o)
        assert e.value.status == B.DCN_ERR_SHAPE, name


def test_no_wait_ran_out():
    assert B.dcn_wait_timeouts() == 0
