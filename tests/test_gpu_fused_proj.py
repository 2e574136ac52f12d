"""The forward with DCNv4's merged offset/mask projection in the same launch
(dcn_core_fwd_proj) against the oracle's composition: the projection
(oracle/proj.py, binary64) and the core op on the merged rows.

The rows the kernel computes are checked element by element against the
oracle's projection within the a-priori rounding bound of a float32 sum
rounded once, and bit for bit against the separate projection (dcn_linear);
the output is checked against the oracle's forward on those rows.  Outputs
sit between canary guards."""
import math

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

ROUND = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def _layer(w, K: int, rs: int, seed: int = 3):
    """Features U(-1, 1) and a layer whose offset rows give offsets of about
    the workload's offset spread, its mask rows about N(0, 1) values."""
    g = torch.Generator().manual_seed(seed)
    dt = DTYPES[w.dtype]
    feat = (torch.rand(w.N, w.H_out, w.W_out, K, generator=g) * 2 - 1).to(dt)
    scale = torch.full((w.G * rs,), math.sqrt(3.0))
    for grp in range(w.G):
        scale[grp * rs:grp * rs + 2 * w.P] *= w.offset_std
    wt = (torch.randn(w.G * rs, K, generator=g) / math.sqrt(K) * scale[:, None]).to(dt)
    b = (0.1 * torch.randn(w.G * rs, generator=g)).to(dt)
    return feat, wt, b


def _run(w, inp, feat, wt, b, rs, with_rows=True):
    dt = DTYPES[w.dtype]
    out = Guarded((w.N, w.H_out, w.W_out, w.C), dt)
    rows = Guarded((w.N, w.H_out, w.W_out, w.G, rs), dt) if with_rows else None
    B.dcn_core_fwd_proj(lib_params(w), inp.cuda(), feat.cuda(), wt.cuda(),
                        b.cuda() if b is not None else None, rs, out.t,
                        rows.t if rows is not None else None)
    torch.cuda.synchronize()
    out.check("output")
    if rows is not None:
        rows.check("offset_mask")
    return out.t, rows.t if rows is not None else None


def _check(w, K, rs, bias=True, seed=3, same_kernel=True):
    inp = make_inputs(w)["input"]
    feat, wt, b = _layer(w, K, rs, seed)
    if not bias:
        b = None
    out, rows = _run(w, inp, feat, wt, b, rs)
    # the rows: the oracle's projection within the rounding bound, and the
    # separate projection bit for bit
    x = f64(feat).reshape(-1, K)
    ref = proj.linear(x, f64(wt), f64(b) if b is not None else None)
    got = f64(rows).reshape(ref.shape)
    mag = np.abs(x) @ np.abs(f64(wt)).T + (np.abs(f64(b))[None, :] if b is not None else 0)
    bound = ROUND[w.dtype] * np.abs(ref) + (K + 2) * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound), f"{w.name}: rows outside the rounding bound"
    sep = B.linear(feat.cuda().reshape(-1, K), wt.cuda(), b.cuda() if b is not None else None)
    assert torch.equal(sep.reshape(rows.shape), rows), f"{w.name}: rows differ from dcn_linear's"
    # the output: the oracle's forward on the same rows
    r = f64(rows)
    off = r[..., :2 * w.P].reshape(w.N, w.H_out, w.W_out, w.G, w.P, 2)
    msk = r[..., 2 * w.P:3 * w.P]
    expect = oracle.forward(oracle_params(w), f64(inp), np.ascontiguousarray(off),
                            np.ascontiguousarray(msk))
    assert_close(out, expect, w.dtype, f"{w.name} fused output")
    # the same launch without writing the rows gives the same output; when
    # the call takes another kernel without them, that output meets the oracle
    # on the same rows
    out2, _ = _run(w, inp, feat, wt, b, rs, with_rows=False)
    if same_kernel:
        assert torch.equal(out, out2)
    else:
        assert_close(out2, expect, w.dtype, f"{w.name} single-launch output")
    return out


# FlashInternImage-T stages (DCNv4, gc 16, 9 points, rows of 32) at two
# images, and InternImage-G stage 1 (DCNv3 softmax, gc 32; 9 points in rows
# of 32, 8 points without the centre in rows of 24) at one
STAGES = [("t_stage1_f16", 2, 64), ("t_stage2_bf16", 2, 128), ("t_stage3_bf16", 2, 256),
          ("t_stage4_bf16", 4, 256), ("g_stage1_bf16", 1, 256), ("g_stage1_rc_bf16", 1, 128)]


# the persistent, warp-specialised kernel (where its buffers fit) and the
# per-tile kernel
# (the fwd_proj switch at 2 keeps the single launch although offset_mask is
# given, so that its rows can be checked)
KERNELS = {"persistent": {"fwd_proj": 2}, "per_tile": {"fwd_proj": 2, "fwd_proj_ws": 0}}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name,N,K", STAGES, ids=[s[0] for s in STAGES])
def test_stage_shapes(name, N, K, kernel, opts):
    opts.update(KERNELS[kernel])
    w = WORKLOADS[name].with_(N=N)
    _check(w, K, 24 if w.P == 8 else 32)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("K", [64, 128, 192, 256])
@pytest.mark.parametrize("sm,rc", [(0, 0), (1, 0), (1, 1)])
def test_ragged_tiles(dt, K, sm, rc, kernel, opts):
    opts.update(KERNELS[kernel])
    # 9 x 13 pixels: ragged tiles in both directions (rows of the projection's
    # tile past the image are computed and dropped)
    w = small(f"fp_{dt}_{K}_{sm}{rc}", dt, gc=16, G=4, N=2, H=9, W=13, softmax=sm,
              remove_center=rc, offset_std=2.0)
    _check(w, K, 24 if w.P == 8 else 32, seed=K + sm)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("gc,G,rs", [(8, 8, 32), (32, 2, 40), (16, 8, 48)])
def test_group_blocks_and_row_strides(gc, G, rs, kernel, opts):
    opts.update(KERNELS[kernel])
    # several blocks per tile's groups (each projects its own groups' rows),
    # wider rows than 3P
    w = small(f"fp_g{gc}_{G}_{rs}", "bf16", gc=gc, G=G, N=2, H=12, W=10, offset_std=2.5)
    _check(w, 64, rs)


def test_no_bias(opts):
    opts.set("fwd_proj", 2)
    w = small("fp_nobias", "f16", gc=16, G=4, N=1, H=16, W=16)
    _check(w, 128, 32, bias=False)


def test_plane_smaller_than_tile(opts):
    opts.set("fwd_proj", 2)
    w = small("fp_small", "bf16", gc=16, G=4, N=3, H=3, W=5)
    _check(w, 64, 32)


def test_many_tiles_per_block(opts):
    # 64 images of 56 x 56: each persistent block walks about 21 tiles, so both
    # buffers of every pipeline stage turn over many times
    opts.set("fwd_proj", 2)
    w = WORKLOADS["t_stage1_f16"]
    _check(w, 64, 32)


@pytest.mark.parametrize("name,N,K", [("t_stage1_f16", 2, 64), ("g_stage1_bf16", 1, 256)])
def test_default_policy(name, N, K):
    # by default a call with offset_mask runs the two launches and one without
    # runs the single launch: the same rows, the same output
    w = WORKLOADS[name].with_(N=N)
    _check(w, K, 32, same_kernel=False)


@pytest.mark.parametrize("why", ["switch", "k96", "f32"])
def test_two_launch_fallback(why, opts):
    # outside the single launch (switched off, K not a multiple of 64, float32)
    # the call projects into offset_mask and runs the core on it: same checks;
    # without offset_mask such a call is refused
    dt = "f32" if why == "f32" else "bf16"
    K = 96 if why == "k96" else 64
    if why == "switch":
        opts.set("fwd_proj", 0)
    w = small(f"fp_fb_{why}", dt, gc=16, G=4, N=2, H=11, W=9, offset_std=2.0)
    inp = make_inputs(w)["input"]
    feat, wt, b = _layer(w, K, 32)
    out, rows = _run(w, inp, feat, wt, b, 32)
    r = f64(rows)
    off = r[..., :2 * w.P].reshape(w.N, w.H_out, w.W_out, w.G, w.P, 2)
    expect = oracle.forward(oracle_params(w), f64(inp), np.ascontiguousarray(off),
                            np.ascontiguousarray(r[..., 2 * w.P:3 * w.P]))
    assert_close(out, expect, dt, f"fallback {why}")
    ref = proj.linear(f64(feat).reshape(-1, K), f64(wt), f64(b))
    assert_close(rows, ref.reshape(r.shape), dt, f"fallback {why} rows")
    # without offset_mask the two launches have nowhere to put the rows
    with pytest.raises(B.DCNError) as e:
        _run(w, inp, feat, wt, b, 32, with_rows=False)
    assert e.value.status == B.DCN_ERR_UNSUPPORTED


def test_no_wait_ran_out():
    assert B.dcn_wait_timeouts() == 0
