"""The linear projections around the core (dcn_linear) against the oracle
(oracle/proj.py), on the tensor-core kernels and on the CUDA-core kernel, and
composed with the core op as DCNv4's merged offset/mask projection."""
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


def _data(M, K, N, dt, bias=True, seed=5):
    g = torch.Generator().manual_seed(seed)
    x = (torch.rand(M, K, generator=g) * 2 - 1).to(DT[dt])
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(DT[dt])
    b = torch.randn(N, generator=g).to(DT[dt]) if bias else None
    return x, w, b


# The a-priori error of a float32 dot product of K terms rounded once to the
# storage type: (K + 2) * 2^-24 * sum_k |x_k w_k| (+ |b|) for the float32
# accumulation, plus the unit roundoff of the storage type times the result
# (2^-8 for bfloat16's 8 significant bits, 2^-11 for float16's 11, 2^-24 for
# float32).
ROUND = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}


def _check(M, K, N, dt, bias=True):
    x, w, b = _data(M, K, N, dt, bias)
    y = B.linear(x.cuda(), w.cuda(), b.cuda() if b is not None else None)
    torch.cuda.synchronize()
    ref = proj.linear(f64(x), f64(w), f64(b) if b is not None else None)
    assert_close(y, ref, dt, f"linear {M}x{K}x{N}")
    err = np.abs(f64(y) - ref)
    mag = np.abs(f64(x)) @ np.abs(f64(w)).T + (np.abs(f64(b))[None, :] if b is not None else 0)
    bound = ROUND[dt] * np.abs(ref) + (K + 2) * 2.0 ** -24 * mag
    assert np.all(err <= bound), \
        f"linear {M}x{K}x{N}: element error {err.max():.3e} above the rounding bound"


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_tensor_core_single_tile(dt):
    # one 128-row tile, one 64-channel block, the narrowest output
    _check(128, 64, 16, dt)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M", [1, 127, 129, 1000])
@pytest.mark.parametrize("K,N", [(64, 128), (128, 64), (192, 48), (256, 256), (64, 112)])
@pytest.mark.parametrize("bias", [True, False])
def test_tensor_core_shapes(dt, M, K, N, bias):
    # ragged row counts (the last tile's rows past M are read as zeros and not
    # written), up to four 64-channel blocks and 256 outputs
    _check(M, K, N, dt, bias)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M", [1, 129, 1000])
@pytest.mark.parametrize("K,N", [(320, 64), (512, 512), (1024, 128), (128, 320), (64, 768),
                                 (512, 1024)])
def test_tensor_core_k_loop_shapes(dt, M, K, N):
    # layers whose W does not fit in shared memory: the K loop through (x, W)
    # chunk stages, output tiles of 64 to 256 columns, ragged row counts
    _check(M, K, N, dt)


@pytest.mark.parametrize("bn", ["64", "128"])
def test_tensor_core_k_loop_narrow_tiles(bn, opts):
    # the same layer with its output split into 64- or 128-column tiles
    opts.set("linear_bn", int(bn))
    _check(300, 512, 512, "bf16")


def test_full_size_projection_at_g_stage1():
    # InternImage-G stage 1's 512 -> 512 projections on 2 x 128 x 128 pixels,
    # checked at sampled rows
    M, K, N = 2 * 128 * 128, 512, 512
    x, w, b = _data(M, K, N, "bf16")
    y = B.linear(x.cuda(), w.cuda(), b.cuda())
    torch.cuda.synchronize()
    rows = np.random.default_rng(1).choice(M, 2048, replace=False)
    ref = proj.linear(f64(x[rows]), f64(w), f64(b))
    assert_close(y[torch.from_numpy(rows).cuda()], ref, "bf16", "projection rows")


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("K,N", [(37, 13), (64, 16), (8, 300), (512, 96)])
def test_cuda_core_path(dt, K, N, opts):
    # shapes outside the tensor-core path, float32, and the tensor-core shapes
    # forced onto the CUDA-core kernel
    opts.set("linear_tc", 0)
    _check(77, K, N, dt)


def test_misaligned_rows_take_the_cuda_core_path():
    x, w, b = _data(64, 64, 16, "bf16")
    buf = torch.empty(64 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    xs = buf[1:].view(64, 64)
    xs.copy_(x.cuda())
    y = B.linear(xs, w.cuda(), b.cuda())
    torch.cuda.synchronize()
    assert_close(y, proj.linear(f64(x), f64(w), f64(b)), "bf16", "misaligned x")


def test_full_size_projection_at_t_stage1():
    # FlashInternImage-T stage 1: 64 x 56 x 56 pixels of 64 channels into the
    # merged offset/mask rows (4 groups x 32); checked at sampled rows
    M, K, N = 64 * 56 * 56, 64, 128
    x, w, b = _data(M, K, N, "f16")
    y = B.linear(x.cuda(), w.cuda(), b.cuda())
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(M, 4096, replace=False)
    ref = proj.linear(f64(x[rows]), f64(w), f64(b))
    assert_close(y[torch.from_numpy(rows).cuda()], ref, "f16", "projection rows")


@pytest.mark.parametrize("name,rs", [("t_stage1_f16", 32), ("g_stage1_rc_bf16", 24)])
def test_merged_projection_feeds_the_core(name, rs):
    # DCNv4's module path: features -> one linear layer -> the merged
    # offset/mask tensor -> the core op, against the oracle's projection and
    # core on the same rounded values
    w_ = WORKLOADS[name].with_(N=1)
    t = make_inputs(w_)
    G, P, C = w_.G, w_.P, w_.C
    dt = w_.dtype
    gen = torch.Generator().manual_seed(9)
    feat = (torch.rand(w_.N, w_.H_out, w_.W_out, C, generator=gen) * 2 - 1).to(DT[dt])
    wo = (torch.randn(G * P * 2, C, generator=gen) * 0.5).to(DT[dt])
    wm = (torch.randn(G * P, C, generator=gen) / C ** 0.5).to(DT[dt])
    bo = torch.randn(G * P * 2, generator=gen).to(DT[dt])
    bm = torch.randn(G * P, generator=gen).to(DT[dt])
    wmerged, bmerged = proj.merged_weights(f64(wo), f64(bo), f64(wm), f64(bm), G, P, rs)
    wmt = torch.from_numpy(wmerged).to(DT[dt])
    bmt = torch.from_numpy(bmerged).to(DT[dt])
    om = B.linear(feat.cuda(), wmt.cuda(), bmt.cuda())        # (N, Ho, Wo, G*rs)
    out = torch.empty(w_.N, w_.H_out, w_.W_out, C, dtype=DT[dt], device="cuda")
    B.dcn_core_fwd_om(lib_params(w_), t["input"].cuda(), om.contiguous(), rs, out)
    torch.cuda.synchronize()
    # the oracle: the projection in binary64, rounded to the storage type as
    # the GPU's is, then the core op on those values
    ref_om = proj.linear(f64(feat.reshape(-1, C)), wmerged, bmerged)
    assert_close(om.reshape(-1, G * rs), ref_om, dt, "offset_mask")
    om_r = om.float().cpu().reshape(w_.N, w_.H_out, w_.W_out, G, rs).double().numpy()
    off = om_r[..., :2 * P].reshape(w_.N, w_.H_out, w_.W_out, G, P, 2)
    msk = om_r[..., 2 * P:3 * P]
    ref = oracle.forward(oracle_params(w_), f64(t["input"]), off, msk)
    assert_close(out, ref, dt, "core on the projected offsets")


def test_no_tensor_core_wait_ran_out():
    assert B.dcn_wait_timeouts() == 0
