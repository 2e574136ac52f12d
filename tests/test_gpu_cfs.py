"""The centre feature scale (dcn_center_feature_scale / _bwd) against the
oracle (oracle/proj.py), through the C ABI: every vector width and the
per-group kernel, ragged row counts, in-place calls, and the gate composed with
the core op and the gate's projection at FlashInternImage-T stage 1's shape."""
import numpy as np
import pytest
import torch

import oracle
from oracle import proj
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import WORKLOADS, make_inputs
from parity import assert_close, f64, lib_params, oracle_params

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native", "oracle_lib")]

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
# unit roundoff of the storage type (one rounding of each result), and half
# its smallest subnormal spacing: results below the normal range round with
# that absolute error instead
ROUND = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}
ETA = {"bf16": 2.0 ** -134, "f16": 2.0 ** -25, "f32": 2.0 ** -150}


def _data(M, C, G, dt, seed=11):
    g = torch.Generator().manual_seed(seed)
    core = (torch.rand(M, C, generator=g) * 4 - 2).to(DT[dt])
    x = (torch.rand(M, C, generator=g) * 4 - 2).to(DT[dt])
    l = (torch.randn(M, G, generator=g) * 3).to(DT[dt])
    go = torch.randn(M, C, generator=g).to(DT[dt])
    return core, x, l, go


def _nan(shape, dt, extra=0):
    """A NaN-filled device buffer; extra > 0 shifts it by that many elements."""
    buf = torch.full((int(np.prod(shape)) + extra,), float("nan"), dtype=DT[dt], device="cuda")
    return buf[extra:].view(*shape)


def _fwd_bound(core, x, ref, dt):
    # one rounding of the result, plus float32 error of the gate and the FMA
    return ROUND[dt] * np.abs(ref) + ETA[dt] + 2.0 ** -20 * (np.abs(f64(core)) + np.abs(f64(x)))


def _check_fwd(core, x, l, out, G, dt):
    ref = proj.center_feature_scale(f64(core), f64(x), f64(l), G)
    assert_close(out, ref, dt, "centre feature scale")
    err = np.abs(f64(out) - ref)
    assert np.all(err <= _fwd_bound(core, x, ref, dt)), f"max err {err.max():.3e}"


def _check_bwd(go, core, x, l, gcore, gx, gl, G, dt):
    rc, rx, rl = proj.center_feature_scale_backward(f64(go), f64(core), f64(x), f64(l), G)
    for name, got, ref in (("grad_core", gcore, rc), ("grad_x_proj", gx, rx),
                           ("grad_logits", gl, rl)):
        assert_close(got, ref, dt, name)
    g = np.abs(f64(go))
    for got, ref in ((gcore, rc), (gx, rx)):
        err = np.abs(f64(got) - ref)
        assert np.all(err <= ROUND[dt] * np.abs(ref) + ETA[dt] + 2.0 ** -20 * g)
    # the logit gradient sums gc products in float32: (gc + 8) * 2^-24 of the
    # sum of magnitudes, times s (1 - s) <= 1/4, plus the gate's own error
    M, C = core.shape
    gc = C // G
    mag = (g * (np.abs(f64(x)) + np.abs(f64(core)))).reshape(M, G, gc).sum(axis=2)
    err = np.abs(f64(gl) - rl)
    assert np.all(err <= ROUND[dt] * np.abs(rl) + ETA[dt] + (gc + 8) * 2.0 ** -22 * mag)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M", [1, 37, 1000])
@pytest.mark.parametrize("C,G", [(64, 4), (16, 16), (12, 4), (96, 2), (256, 8), (48, 1),
                                 (1024, 2)])
def test_forward_and_backward(dt, M, C, G):
    # gc = 16, 1, 3, 48, 32, 48, 512: 16-byte, 8/4-byte and one-element
    # accesses; gc / V of 1 to 32 lanes, and above 32 (the per-group kernel)
    core, x, l, go = _data(M, C, G, dt)
    cd, xd, ld, god = (t.cuda() for t in (core, x, l, go))
    out = _nan((M, C), dt)
    B.dcn_center_feature_scale(cd, xd, ld, out, G)
    gcore, gx, gl = _nan((M, C), dt), _nan((M, C), dt), _nan((M, G), dt)
    B.dcn_center_feature_scale_bwd(god, cd, xd, ld, gcore, gx, gl, G)
    torch.cuda.synchronize()
    _check_fwd(core, x, l, out, G, dt)
    _check_bwd(go, core, x, l, gcore, gx, gl, G, dt)


@pytest.mark.parametrize("dt", ["f16", "f32"])
@pytest.mark.parametrize("shift", [1, 2, 4])
def test_misaligned_buffers_take_narrower_accesses(dt, shift):
    # buffers one, two or four elements off a 16-byte boundary
    M, C, G = 50, 64, 4
    core, x, l, go = _data(M, C, G, dt, seed=12)
    cd, xd, god = _nan((M, C), dt, shift), _nan((M, C), dt, shift), _nan((M, C), dt, shift)
    cd.copy_(core)
    xd.copy_(x)
    god.copy_(go)
    ld = l.cuda()
    out = _nan((M, C), dt, shift)
    B.dcn_center_feature_scale(cd, xd, ld, out, G)
    gcore, gx, gl = _nan((M, C), dt, shift), _nan((M, C), dt, shift), _nan((M, G), dt)
    B.dcn_center_feature_scale_bwd(god, cd, xd, ld, gcore, gx, gl, G)
    torch.cuda.synchronize()
    _check_fwd(core, x, l, out, G, dt)
    _check_bwd(go, core, x, l, gcore, gx, gl, G, dt)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_in_place(dt):
    M, C, G = 300, 64, 4
    core, x, l, go = _data(M, C, G, dt, seed=13)
    # out over core, then out over x_proj
    cd, xd, ld = core.cuda(), x.cuda(), l.cuda()
    B.dcn_center_feature_scale(cd, xd, ld, cd, G)
    xd2 = x.cuda()
    B.dcn_center_feature_scale(core.cuda(), xd2, ld, xd2, G)
    # grad_core over grad_out
    god = go.cuda()
    gx, gl = _nan((M, C), dt), _nan((M, G), dt)
    B.dcn_center_feature_scale_bwd(god, core.cuda(), x.cuda(), ld, god, gx, gl, G)
    torch.cuda.synchronize()
    _check_fwd(core, x, l, cd, G, dt)
    _check_fwd(core, x, l, xd2, G, dt)
    _check_bwd(go, core, x, l, god, gx, gl, G, dt)


def test_saturated_gates_pass_one_side_exactly():
    # logits of +-60 give s = 1 or 0 in float32: the output is x_proj or the
    # core's output, bit for bit
    M, C, G = 64, 64, 4
    core, x, _, _ = _data(M, C, G, "f16", seed=14)
    l = torch.full((M, G), 60.0, dtype=torch.float16)
    l[:, ::2] = -60.0
    out = B.center_feature_scale(core.cuda(), x.cuda(), l.cuda()).cpu()
    gc = C // G
    for g in range(G):
        side = core if g % 2 == 0 else x
        assert torch.equal(out[:, g * gc:(g + 1) * gc], side[:, g * gc:(g + 1) * gc])


def test_full_size_at_t_stage1():
    # FlashInternImage-T stage 1: 64 x 56 x 56 pixels of 64 channels, 4 groups
    M, C, G = 64 * 56 * 56, 64, 4
    core, x, l, go = _data(M, C, G, "f16", seed=15)
    cd, xd, ld, god = (t.cuda() for t in (core, x, l, go))
    out = B.center_feature_scale(cd, xd, ld)
    gcore, gx, gl = B.center_feature_scale_backward(god, cd, xd, ld)
    torch.cuda.synchronize()
    _check_fwd(core, x, l, out, G, "f16")
    _check_bwd(go, core, x, l, gcore, gx, gl, G, "f16")


@pytest.mark.parametrize("name", ["t_stage1_f16", "g_stage1_bf16"])
def test_gate_after_the_core(name):
    # the module's tail at stride 1: the core's output, the gate's logits from
    # a linear layer of G outputs, and the mix with the core's own input
    w_ = WORKLOADS[name].with_(N=1)
    t = make_inputs(w_)
    dt = w_.dtype
    C, G = w_.C, w_.G
    gen = torch.Generator().manual_seed(21)
    feat = (torch.rand(w_.N, w_.H_out, w_.W_out, C, generator=gen) * 2 - 1).to(DT[dt])
    wc = (torch.randn(G, C, generator=gen) / C ** 0.5).to(DT[dt])
    bc = torch.randn(G, generator=gen).to(DT[dt])
    core = torch.empty(w_.N, w_.H_out, w_.W_out, C, dtype=DT[dt], device="cuda")
    B.dcn_core_fwd(lib_params(w_), t["input"].cuda(), t["offset"].cuda(), t["mask"].cuda(), core)
    logits = B.linear(feat.cuda(), wc.cuda(), bc.cuda())
    out = B.center_feature_scale(core, t["input"].cuda(), logits)
    torch.cuda.synchronize()
    # the oracle on the values the GPU had: its core output and logits, rounded
    ref_core = oracle.forward(oracle_params(w_), f64(t["input"]), f64(t["offset"]),
                              f64(t["mask"]))
    assert_close(core, ref_core, dt, "core")
    ref_l = proj.linear(f64(feat.reshape(-1, C)), f64(wc), f64(bc))
    assert_close(logits.reshape(-1, G), ref_l, dt, "gate logits")
    ref = proj.center_feature_scale(f64(core.reshape(-1, C)), f64(t["input"].reshape(-1, C)),
                                    f64(logits.reshape(-1, G)), G)
    assert_close(out.reshape(-1, C), ref, dt, "gated output")
