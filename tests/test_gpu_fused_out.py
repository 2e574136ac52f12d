"""The core forward with the output projection (dcn_core_fwd_out), with and
without the centre feature scale between them, against the oracle's
composition: the core op (oracle.forward, binary64), the gate
(oracle/proj.py center_feature_scale, x_proj the core's input), rounding to
the storage type as the core's output is stored, then the projection
(oracle/proj.py linear).

The single launch (the projection on the tensor cores in the forward's
epilogue) is also compared with the two launches through scratch (the core's
output stored, then dcn_linear): the same products of the same rounded values.
Outputs sit between canary guards."""
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


def _layer(w, n_out, seed=9, bias=True):
    g = torch.Generator().manual_seed(seed)
    dt = DTYPES[w.dtype]
    wt = (torch.randn(n_out, w.C, generator=g) / w.C ** 0.5).to(dt)
    b = (0.1 * torch.randn(n_out, generator=g)).to(dt) if bias else None
    lg = (torch.randn(w.N, w.H_out, w.W_out, w.G, generator=g) * 2).to(dt)
    return wt, b, lg


def _run(w, t, wt, b, lg, scratch=True, want_scratch=False):
    dt = DTYPES[w.dtype]
    y = Guarded((w.N, w.H_out, w.W_out, wt.shape[0]), dt)
    sc = Guarded((w.N, w.H_out, w.W_out, w.C), dt) if scratch else None
    B.dcn_core_fwd_out(lib_params(w), t["input"].cuda(), t["offset"].cuda(), t["mask"].cuda(),
                       lg.cuda() if lg is not None else None, wt.cuda(),
                       b.cuda() if b is not None else None, y.t, sc.t if sc is not None else None)
    torch.cuda.synchronize()
    y.check("y")
    if sc is not None:
        sc.check("scratch")
    return (y.t, sc.t if sc is not None else None) if want_scratch else y.t


def _expect(w, t, wt, b, lg):
    out = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    M = w.N * w.H_out * w.W_out
    out = out.reshape(M, w.C)
    if lg is not None:
        out = proj.center_feature_scale(out, f64(t["input"]).reshape(M, w.C),
                                        f64(lg).reshape(M, w.G), w.G)
    # the core's output as stored: rounded to the storage type
    stored = torch.from_numpy(out).to(DTYPES[w.dtype]).double().numpy()
    y = proj.linear(stored, f64(wt), f64(b) if b is not None else None)
    return y.reshape(w.N, w.H_out, w.W_out, wt.shape[0])


def _check(w, n_out, opts, gate=True, bias=True, seed=9):
    t = make_inputs(w)
    wt, b, lg = _layer(w, n_out, seed, bias)
    lg = lg if gate else None
    ref = _expect(w, t, wt, b, lg)
    fused = _run(w, t, wt, b, lg, scratch=False)
    assert_close(fused, ref, w.dtype, f"{w.name} single launch")
    opts.set("fwd_out", 0)
    two = _run(w, t, wt, b, lg)
    opts.set("fwd_out", 1)
    assert_close(two, ref, w.dtype, f"{w.name} two launches")
    # the same rounded inputs and products: at most one rounding step apart
    u = ROUND[w.dtype]
    d = np.abs(f64(fused) - f64(two))
    assert np.all(d <= 2 * u * np.abs(f64(two)) + 1e-30 + u * np.abs(ref).max() * 2 ** -4), \
        f"{w.name}: single and two launches differ by {d.max()}"
    return fused


# FlashInternImage-T stage 1 (C = 64 in 4 groups of 16) at two images, both
# 16-bit types, with and without the gate and the bias, n_out of 64 (the
# module's output projection) and 16 / 128
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("n_out", [64, 16, 128])
@pytest.mark.parametrize("gate,bias", [(True, True), (False, True), (True, False)])
def test_stage1_shape(dt, n_out, gate, bias, opts):
    w = WORKLOADS["t_stage1_f16"].with_(N=2, dtype=dt)
    _check(w, n_out, opts, gate, bias)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("gc,G", [(16, 4), (8, 8), (32, 2)])
@pytest.mark.parametrize("sm,rc", [(0, 0), (1, 0), (1, 1)])
def test_ragged_planes(dt, gc, G, sm, rc, opts):
    # 13 x 11 pixels (ragged tiles) of 64 channels in 4 / 8 / 2 groups (16-,
    # 8- and 16-channel slices), softmax and centre removal; offsets N(0, 3)
    w = small(f"out_{dt}_{gc}_{G}_{sm}{rc}", dt, gc=gc, G=G, N=2, H=13, W=11, softmax=sm,
              remove_center=rc, offset_std=3.0)
    _check(w, 64, opts, seed=gc + G)


@pytest.mark.parametrize("k", [5, 7])
def test_large_kernels(k, opts):
    # 5 x 5 and 7 x 7 taps (the 7 x 7 window takes the larger shared-memory
    # budget, with the epilogue's operand tiles after it)
    w = small(f"out_k{k}", "f16", gc=16, G=4, N=2, H=13, W=11, kernel_h=k, kernel_w=k,
              pad_h=k // 2, pad_w=k // 2, softmax=1)
    _check(w, 64, opts, seed=k)


def test_many_tiles_per_sm(opts):
    # 64 images of 56 x 56: every SM runs many blocks, each allocating and
    # freeing its tensor memory
    _check(WORKLOADS["t_stage1_f16"], 64, opts)


def test_scratch_selects_the_way(opts):
    # with scratch the two launches (scratch then holds the core's output with
    # the gate, as dcn_core_fwd_cfs stores it); with the fwd_out switch at 2
    # the single launch even with scratch, which it leaves untouched
    w = WORKLOADS["t_stage1_f16"].with_(N=2)
    t = make_inputs(w)
    wt, b, lg = _layer(w, 64)
    single = _run(w, t, wt, b, lg, scratch=False)
    y, sc = _run(w, t, wt, b, lg, want_scratch=True)
    core = torch.empty_like(sc)
    B.dcn_core_fwd_cfs(lib_params(w), t["input"].cuda(), t["offset"].cuda(), t["mask"].cuda(),
                       lg.cuda(), core)
    torch.cuda.synchronize()
    assert torch.equal(sc, core)
    opts.set("fwd_out", 0)
    assert torch.equal(y, _run(w, t, wt, b, lg))
    opts.set("fwd_out", 2)
    y2, sc2 = _run(w, t, wt, b, lg, want_scratch=True)
    assert torch.equal(y2, single)
    assert bool(torch.all(torch.isnan(sc2))), "the single launch wrote scratch"


@pytest.mark.parametrize("why", ["c128", "f32", "n_out_24"])
def test_two_launch_fallback(why, opts):
    # 128 channels, float32 storage or an n_out that is not a multiple of 16:
    # the two launches through scratch, and DCN_ERR_UNSUPPORTED without it
    if why == "c128":
        w = small("out_fb_c128", "bf16", gc=16, G=8, N=2, H=9, W=10)
    elif why == "f32":
        w = small("out_fb_f32", "f32", gc=16, G=4, N=2, H=9, W=10)
    else:
        w = small("out_fb_n24", "f16", gc=16, G=4, N=2, H=9, W=10)
    n_out = 24 if why == "n_out_24" else 64
    t = make_inputs(w)
    wt, b, lg = _layer(w, n_out)
    assert_close(_run(w, t, wt, b, lg), _expect(w, t, wt, b, lg), w.dtype, f"fallback {why}")
    with pytest.raises(B.DCNError) as e:
        _run(w, t, wt, b, lg, scratch=False)
    assert e.value.status == B.DCN_ERR_UNSUPPORTED


def test_argument_errors():
    w = small("out_err", "f16", gc=16, G=4, N=1, H=9, W=9)
    t = {k: v.cuda() for k, v in make_inputs(w).items()}
    wt, b, lg = (x.cuda() for x in _layer(w, 64))
    y = torch.empty(w.N, w.H_out, w.W_out, 64, dtype=torch.float16, device="cuda")
    p = lib_params(w)
    with pytest.raises(B.DCNError) as e:
        B.dcn_core_fwd_out(p, t["input"], t["offset"], t["mask"], lg, wt, b, None)
    assert e.value.status == B.DCN_ERR_NULL
    with pytest.raises(B.DCNError) as e:
        B.dcn_core_fwd_out(p, t["input"], t["offset"], t["mask"], lg, wt[:0], b, y)
    assert e.value.status == B.DCN_ERR_SHAPE
    # the gate needs an output the input's size
    v = small("out_err_s2", "f16", gc=16, G=4, N=1, H=9, W=9, stride_h=2, stride_w=2)
    tv = {k: x.cuda() for k, x in make_inputs(v).items()}
    lv = _layer(v, 64)[2].cuda()
    yv = torch.empty(v.N, v.H_out, v.W_out, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(B.DCNError) as e:
        B.dcn_core_fwd_out(lib_params(v), tv["input"], tv["offset"], tv["mask"], lv, wt, b, yv)
    assert e.value.status == B.DCN_ERR_SHAPE


def test_empty_batch():
    # no units: nothing is read or written, every pointer may be NULL
    w = small("out_empty", "f16", gc=16, G=4, N=0)
    B.dcn_core_fwd_out(lib_params(w), None, None, None, None,
                       torch.empty(64, 64, dtype=torch.float16, device="cuda"), None, None)


def test_no_wait_ran_out():
    assert B.dcn_wait_timeouts() == 0
