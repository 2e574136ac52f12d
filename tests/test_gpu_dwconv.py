"""The offset branch's feature step (dcn_dwconv_ln_gelu: depthwise k x k
convolution, LayerNorm over the channels, exact GELU) against the oracle
(oracle/dwconv.py), on the tiled kernel at every patch layout and on the
one-warp-per-pixel kernel, at the FlashInternImage-T and InternImage-G shapes
and on ragged and degenerate cases.  Outputs sit between canary guards."""
import numpy as np
import pytest
import torch

from oracle import dwconv as odw
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import make_dwconv_inputs
from parity import Guarded, assert_close, f64

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native")]


def _run(t: dict, eps: float, dev="cuda"):
    x = t["x"].to(dev)
    y = Guarded(tuple(x.shape), x.dtype, dev)
    bias = t["bias"].to(dev) if t["bias"] is not None else None
    B.dcn_dwconv_ln_gelu(x, t["weight"].to(dev), bias, t["gamma"].to(dev), t["beta"].to(dev),
                         y.t, eps)
    torch.cuda.synchronize()
    y.check("dwconv_ln_gelu")
    return y.t


def _ref(t: dict, eps: float, images=None):
    x = f64(t["x"]) if images is None else f64(t["x"][images])
    b = f64(t["bias"]) if t["bias"] is not None else np.zeros(x.shape[-1])
    return odw.dwconv_ln_gelu(x, f64(t["weight"]), b, f64(t["gamma"]), f64(t["beta"]), eps)


def _check(N, H, W, C, k, dt, eps=1e-6, bias=True, seed=0, images=None):
    t = make_dwconv_inputs(N, H, W, C, k, dt, seed=seed, bias=bias)
    y = _run(t, eps)
    got = y if images is None else y[images]
    assert_close(got, _ref(t, eps, images), dt, f"dwconv {N}x{H}x{W}x{C} k{k} {dt}")


# FlashInternImage-T stages (channels 64 doubling per stage at 56/28/14/7
# pixels, batch 64) and the InternImage-G first stage (512 channels at
# 128 x 128, batch 2), kernel 5; the oracle checks whole images.
@pytest.mark.parametrize("N,H,C,dt,images", [
    (64, 56, 64, "f16", [0, 37, 63]),
    (64, 28, 128, "bf16", [5, 63]),
    (64, 14, 256, "bf16", [0, 63]),
    (64, 7, 512, "f16", [1, 62]),
    (2, 128, 512, "bf16", [1]),
])
def test_stage_shapes(N, H, C, dt, images):
    _check(N, H, H, C, 5, dt, images=images)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("C", [64, 128, 192, 256, 512])  # 192: the general kernel
@pytest.mark.parametrize("k", [3, 5])
def test_tiled_ragged(opts, dt, C, k):
    # 9 x 13 pixels: every tile layout ends in a ragged tile in both directions
    _check(2, 9, 13, C, k, dt, seed=C + k)


@pytest.mark.parametrize("patches", [1, 2, 4, 8])
@pytest.mark.parametrize("py", [2, 4])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("k", [3, 5])
def test_tiled_patch_layouts(opts, patches, py, dt, k):
    # at C = 64 a block takes 1, 2, 4 or 8 patches (1 x 1 to 2 x 4) of 4 or 2
    # rows, each forced here.  10 images of 11 x 18
    # pixels make more tiles than a block count that fills the GPU once only
    # at the smallest tiles, so the persistent blocks take several tiles each.
    opts.set("dw_patches", patches)
    opts.set("dw_py", py)
    _check(10, 11, 18, 64, k, dt, seed=patches + py, images=[0, 4, 9])


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_tiles_per_block(dt):
    # far more tiles than resident blocks (64 images of 56 x 56 at 64
    # channels: 1792 tiles of 8 x 16), the double-buffered staging turns over
    # many times in each block; every image is checked
    _check(64, 56, 56, 64, 5, dt, seed=11)


@pytest.mark.parametrize("dt", ["f32", "f16"])
@pytest.mark.parametrize("C,k", [(64, 5), (80, 3), (3, 5), (33, 7), (512, 1), (96, 9)])
def test_general_kernel(opts, dt, C, k):
    # shapes outside the tiled kernel, and the tiled kernel's shapes forced onto
    # the general one
    if C % 64 == 0 and k in (3, 5):
        opts.set("dw_tiled", 0)
    _check(2, 7, 10, C, k, dt, seed=C * k)


@pytest.mark.parametrize("dt,C", [("f32", 512), ("f16", 1024), ("bf16", 2048)])
def test_widest_channels(dt, C):
    # 512 float32 channels: one 2 x 4 patch per block, one block per SM; wider:
    # the general kernel
    _check(2, 6, 9, C, 5, dt, seed=C)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("H,W", [(1, 1), (1, 40), (40, 1), (2, 3)])
def test_small_images(dt, H, W):
    # images smaller than the kernel: most taps fall outside
    _check(3, H, W, 64, 5, dt, seed=H * 64 + W)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_no_bias_and_eps(dt):
    _check(2, 9, 9, 128, 5, dt, bias=False, eps=1e-5)
    _check(2, 9, 9, 128, 5, dt, eps=0.5)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("C", [64, 80])
def test_constant_features_give_gelu_of_beta(dt, C):
    # a zero kernel and a constant bias make every pixel's C sums equal: the
    # variance is zero, LayerNorm returns beta and the output is GELU(beta)
    t = make_dwconv_inputs(2, 5, 6, C, 5, dt, seed=3)
    t["weight"] = torch.zeros_like(t["weight"])
    t["bias"] = torch.full_like(t["gamma"], 0.75)
    y = _run(t, 1e-6)
    ref = odw.gelu(np.broadcast_to(f64(t["beta"]), (2, 5, 6, C)))
    assert_close(y, ref, dt, "constant features")


def test_no_images_launches_nothing():
    t = make_dwconv_inputs(1, 4, 4, 64, 5, "bf16")
    x = torch.empty((0, 4, 4, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    B.dcn_dwconv_ln_gelu(x, t["weight"].cuda(), t["bias"].cuda(), t["gamma"].cuda(),
                         t["beta"].cuda(), y, 1e-6)
    torch.cuda.synchronize()


def test_torch_facing_wrapper():
    t = make_dwconv_inputs(2, 12, 12, 128, 5, "bf16", seed=9)
    y = B.dwconv_ln_gelu(t["x"].cuda(), t["weight"].cuda(), t["bias"].cuda(), t["gamma"].cuda(),
                         t["beta"].cuda(), eps=1e-6)
    torch.cuda.synchronize()
    assert_close(y, _ref(t, 1e-6), "bf16", "dwconv_ln_gelu wrapper")
