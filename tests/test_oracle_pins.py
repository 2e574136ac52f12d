"""Pins of the oracle to things other than itself (CPU only).

Every check here compares the oracle with a library routine (``F.unfold``,
``F.grid_sample`` and autograd), with a closed form, with finite differences
or with an invariant.  Between them a dropped term, a wrong sign, a wrong index
or a transposed operand anywhere in the oracle fails at least one check.

The geometry follows the walkthrough of dcnv3_core_pytorch on the page
"没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 四.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import Params

pytestmark = pytest.mark.usefixtures("oracle_lib")


# --------------------------------------------------------------------------
# helpers built from library routines and definitions (not from the oracle)

def unfold_taps(x_nhwc: np.ndarray, p: Params) -> np.ndarray:
    """im2col of a standard strided / dilated / padded convolution.

    Returns (N, Ho, Wo, kh, kw, C): the input value that the (ky, kx) tap of a
    plain convolution reads for each output pixel, zero in the padding.
    """
    x = torch.from_numpy(np.ascontiguousarray(x_nhwc)).permute(0, 3, 1, 2)
    N, C, H, W = x.shape
    cols = F.unfold(x, (p.kernel_h, p.kernel_w), dilation=(p.dilation_h, p.dilation_w),
                    padding=(p.pad_h, p.pad_w), stride=(p.stride_h, p.stride_w))
    ho, wo = oracle.out_shape(p)
    cols = cols.reshape(N, C, p.kernel_h, p.kernel_w, ho, wo)
    return cols.permute(0, 4, 5, 2, 3, 1).numpy()


def tap_index(p: Params, ix: int, iy: int) -> int:
    """Position of kernel tap (ix, iy) in the P points: x-major, centre removed."""
    k = ix * p.kernel_h + iy
    c = (p.kernel_w - 1) // 2 * p.kernel_h + (p.kernel_h - 1) // 2
    if p.remove_center:
        assert k != c
        if k > c:
            k -= 1
    return k


def shift(x_nhwc: np.ndarray, dx: int, dy: int) -> np.ndarray:
    """y[n, i, j] = x[n, i + dy, j + dx], zero where that falls outside."""
    y = np.zeros_like(x_nhwc)
    N, H, W, C = x_nhwc.shape
    for i in range(H):
        for j in range(W):
            si, sj = i + dy, j + dx
            if 0 <= si < H and 0 <= sj < W:
                y[:, i, j] = x_nhwc[:, si, sj]
    return y


def shifted_taps(x_nhwc: np.ndarray, p: Params, dx: int, dy: int) -> np.ndarray:
    """unfold_taps of the zero-padded input translated by (dx, dy): what each
    convolution tap reads after its location moves by whole pixels.  The
    translation acts on the padded frame, so pixels of the image that a moved
    tap reaches from the padding border are kept."""
    xp = np.pad(x_nhwc, ((0, 0), (p.pad_h, p.pad_h), (p.pad_w, p.pad_w), (0, 0)))
    q = Params(**{**p.__dict__, "H": xp.shape[1], "W": xp.shape[2], "pad_h": 0, "pad_w": 0})
    return unfold_taps(shift(xp, dx, dy), q)


def shapes(p: Params):
    ho, wo = oracle.out_shape(p)
    P = oracle.num_points(p)
    return ho, wo, P


def one_hot_mask(p: Params, k: int, ho: int, wo: int, P: int) -> np.ndarray:
    """Weights that select point k: 1 / 0 raw, or logits whose softmax is one-hot."""
    if p.softmax:
        m = np.full((p.N, ho, wo, p.G, P), -1e300)
        m[..., k] = 0.0
    else:
        m = np.zeros((p.N, ho, wo, p.G, P))
        m[..., k] = 1.0
    return m


GEOMS = [
    dict(),
    dict(stride_h=2, stride_w=2),
    dict(dilation_h=2, dilation_w=2, pad_h=2, pad_w=2),
    dict(stride_h=2, stride_w=2, pad_h=1, pad_w=1, dilation_h=2, dilation_w=2),
    dict(kernel_h=1, kernel_w=1, pad_h=0, pad_w=0),
    dict(kernel_h=5, kernel_w=3, pad_h=2, pad_w=0, stride_w=2),
    dict(kernel_h=3, kernel_w=3, pad_h=0, pad_w=3, dilation_w=3),
]


# --------------------------------------------------------------------------
# T1a: zero offsets + one-hot mask reproduce a convolution tap (F.unfold)

@pytest.mark.parametrize("geom", GEOMS)
@pytest.mark.parametrize("softmax", [0, 1])
@pytest.mark.parametrize("coord_f32", [0, 1])
def test_zero_offset_one_hot_is_conv_tap(geom, softmax, coord_f32):
    p = Params(N=2, H=7, W=6, G=2, gc=3, softmax=softmax, coord_f32=coord_f32, **geom)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(1)
    x = rng.uniform(-1, 1, (p.N, p.H, p.W, p.G * p.gc))
    cols = unfold_taps(x, p)
    off = np.zeros((p.N, ho, wo, p.G, P, 2))
    for ix in range(p.kernel_w):
        for iy in range(p.kernel_h):
            k = tap_index(p, ix, iy)
            out = oracle.forward(p, x, off, one_hot_mask(p, k, ho, wo, P))
            np.testing.assert_array_equal(out, cols[:, :, :, iy, ix, :])


def test_remove_center_keeps_order_of_the_other_taps():
    p = Params(N=1, H=6, W=6, G=1, gc=2, remove_center=1)
    ho, wo, P = shapes(p)
    assert P == 8
    assert oracle.taps(p) == [(-1, -1), (-1, 0), (-1, 1), (0, -1), (0, 1), (1, -1), (1, 0), (1, 1)]
    x = np.random.default_rng(2).uniform(-1, 1, (1, 6, 6, 2))
    cols = unfold_taps(x, p)
    off = np.zeros((1, ho, wo, 1, P, 2))
    for ix in range(3):
        for iy in range(3):
            if ix == 1 and iy == 1:
                continue
            out = oracle.forward(p, x, off, one_hot_mask(p, tap_index(p, ix, iy), ho, wo, P))
            np.testing.assert_array_equal(out, cols[:, :, :, iy, ix, :])


# --------------------------------------------------------------------------
# T1b: integer offsets copy pixels exactly; offset_scale scales taps and offsets

@pytest.mark.parametrize("dx,dy", [(1, 0), (0, -2), (3, 2), (-1, -1)])
@pytest.mark.parametrize("coord_f32", [0, 1])
def test_integer_offset_copies_shifted_pixel(dx, dy, coord_f32):
    p = Params(N=1, H=6, W=7, G=2, gc=2, coord_f32=coord_f32)
    ho, wo, P = shapes(p)
    x = np.random.default_rng(3).uniform(-1, 1, (1, 6, 7, 4))
    cols = shifted_taps(x, p, dx, dy)
    off = np.zeros((1, ho, wo, p.G, P, 2))
    off[..., 0] = dx
    off[..., 1] = dy
    for ix in range(3):
        for iy in range(3):
            out = oracle.forward(p, x, off, one_hot_mask(p, tap_index(p, ix, iy), ho, wo, P))
            np.testing.assert_array_equal(out, cols[:, :, :, iy, ix, :])


def test_offset_scale_scales_grid_and_offset():
    # offset_scale 0.5 with dilation 2 puts the taps where dilation 1 puts them,
    # and an offset of 2 then moves the sample by one pixel.
    base = dict(N=1, H=6, W=6, G=1, gc=2)
    p_half = Params(dilation_h=2, dilation_w=2, pad_h=2, pad_w=2, offset_scale=0.5, **base)
    p_one = Params(pad_h=1, pad_w=1, **base)
    assert oracle.out_shape(p_half) == oracle.out_shape(p_one)
    ho, wo, P = shapes(p_one)
    x = np.random.default_rng(4).uniform(-1, 1, (1, 6, 6, 2))
    cols = shifted_taps(x, p_one, 1, -1)
    off = np.zeros((1, ho, wo, 1, P, 2))
    off[..., 0], off[..., 1] = 2.0, -2.0
    for ix in range(3):
        for iy in range(3):
            m = one_hot_mask(p_half, tap_index(p_half, ix, iy), ho, wo, P)
            np.testing.assert_array_equal(oracle.forward(p_half, x, off, m), cols[:, :, :, iy, ix, :])


# --------------------------------------------------------------------------
# T1c: samples pushed out of the image contribute exactly 0 and get no gradient

@pytest.mark.parametrize("far", [20.0, -20.0, 1e30, -1e30, math.inf, -math.inf, math.nan])
@pytest.mark.parametrize("softmax", [0, 1])
def test_out_of_bounds_is_zero(far, softmax):
    p = Params(N=1, H=5, W=5, G=2, gc=3, softmax=softmax)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(5)
    x = rng.uniform(-1, 1, (1, 5, 5, 6))
    off = rng.normal(0, 1, (1, ho, wo, p.G, P, 2))
    off[..., 0] = far
    mask = rng.normal(0, 1, (1, ho, wo, p.G, P))
    out = oracle.forward(p, x, off, mask)
    assert np.all(out == 0.0)
    go = rng.normal(0, 1, out.shape)
    gi, goff, gm = oracle.backward(p, go, x, off, mask)
    assert np.all(gi == 0.0) and np.all(goff == 0.0) and np.all(gm == 0.0)


def test_sample_exactly_at_minus_one_is_dropped():
    # x = -1 exactly: both x-corners are -1 (weight 1, in the padding) and 0
    # (weight 0): the value is 0 either way and the sample is dropped.
    p = Params(N=1, H=3, W=3, G=1, gc=1, kernel_h=1, kernel_w=1, pad_h=0, pad_w=0)
    x = np.arange(1.0, 10.0).reshape(1, 3, 3, 1)
    off = np.zeros((1, 3, 3, 1, 1, 2))
    off[0, :, 0, 0, 0, 0] = -1.0    # wo = 0 -> x = -1
    out = oracle.forward(p, x, off, np.ones((1, 3, 3, 1, 1)))
    assert np.all(out[0, :, 0, 0] == 0.0)
    _, goff, _ = oracle.backward(p, np.ones_like(out), x, off, np.ones((1, 3, 3, 1, 1)))
    assert np.all(goff[0, :, 0] == 0.0)


# --------------------------------------------------------------------------
# T1d: half-pixel offsets give the mean of 2 or 4 neighbours

@pytest.mark.parametrize("coord_f32", [0, 1])
def test_half_pixel_offsets_average_neighbours(coord_f32):
    p = Params(N=1, H=6, W=6, G=2, gc=2, coord_f32=coord_f32)
    ho, wo, P = shapes(p)
    x = np.random.default_rng(6).uniform(-1, 1, (1, 6, 6, 4))
    c00, c01 = shifted_taps(x, p, 0, 0), shifted_taps(x, p, 1, 0)
    c10, c11 = shifted_taps(x, p, 0, 1), shifted_taps(x, p, 1, 1)
    off = np.zeros((1, ho, wo, p.G, P, 2))
    off[..., 0] = 0.5
    for ix in range(3):
        for iy in range(3):
            m = one_hot_mask(p, tap_index(p, ix, iy), ho, wo, P)
            out = oracle.forward(p, x, off, m)
            np.testing.assert_allclose(out, 0.5 * (c00 + c01)[:, :, :, iy, ix], rtol=0, atol=1e-15)
    off[..., 1] = 0.5
    for ix in range(3):
        for iy in range(3):
            m = one_hot_mask(p, tap_index(p, ix, iy), ho, wo, P)
            out = oracle.forward(p, x, off, m)
            want = 0.25 * (c00 + c01 + c10 + c11)[:, :, :, iy, ix]
            np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# T1e: softmax weights sum to one; equal logits average the taps

def test_softmax_weights_sum_to_one():
    p = Params(N=1, H=7, W=7, G=2, gc=2, softmax=1)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(7)
    x = np.full((1, 7, 7, 4), 0.375)
    off = rng.uniform(-0.9, 0.9, (1, ho, wo, p.G, P, 2))
    mask = rng.normal(0, 3, (1, ho, wo, p.G, P))
    out = oracle.forward(p, x, off, mask)
    # interior pixels: every sample lies inside the image, so the output is the
    # constant times the sum of the weights
    np.testing.assert_allclose(out[0, 2:-2, 2:-2], 0.375, rtol=0, atol=1e-15)


def test_softmax_equal_logits_is_mean_of_taps():
    p = Params(N=1, H=6, W=5, G=2, gc=3, softmax=1, stride_h=2)
    ho, wo, P = shapes(p)
    x = np.random.default_rng(8).uniform(-1, 1, (1, 6, 5, 6))
    cols = unfold_taps(x, p)
    out = oracle.forward(p, x, np.zeros((1, ho, wo, p.G, P, 2)), np.full((1, ho, wo, p.G, P), 1.7))
    np.testing.assert_allclose(out, cols.mean(axis=(3, 4)), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# T1f: DCNv4 (no softmax) is linear in the mask

def test_raw_mask_linearity():
    p = Params(N=1, H=6, W=6, G=2, gc=3)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(9)
    x = rng.uniform(-1, 1, (1, 6, 6, 6))
    off = rng.normal(0, 2, (1, ho, wo, p.G, P, 2))
    m1 = rng.normal(0, 1, (1, ho, wo, p.G, P))
    m2 = rng.normal(0, 1, (1, ho, wo, p.G, P))
    o1, o2 = oracle.forward(p, x, off, m1), oracle.forward(p, x, off, m2)
    np.testing.assert_allclose(oracle.forward(p, x, off, 2.5 * m1 - m2), 2.5 * o1 - o2,
                               rtol=0, atol=1e-14)
    assert np.all(oracle.forward(p, x, off, np.zeros_like(m1)) == 0.0)


# --------------------------------------------------------------------------
# T1g: remove_center equals the full kernel with the centre switched off

@pytest.mark.parametrize("softmax", [0, 1])
def test_remove_center_equals_masked_centre(softmax):
    p9 = Params(N=2, H=6, W=6, G=2, gc=3, softmax=softmax)
    p8 = Params(N=2, H=6, W=6, G=2, gc=3, softmax=softmax, remove_center=1)
    ho, wo, P = shapes(p8)
    rng = np.random.default_rng(10)
    x = rng.uniform(-1, 1, (2, 6, 6, 6))
    off8 = rng.normal(0, 2, (2, ho, wo, 2, 8, 2))
    m8 = rng.normal(0, 1, (2, ho, wo, 2, 8))
    off9 = np.insert(off8, 4, 0.0, axis=4)
    m9 = np.insert(m8, 4, -1e300 if softmax else 0.0, axis=4)
    np.testing.assert_allclose(oracle.forward(p8, x, off8, m8), oracle.forward(p9, x, off9, m9),
                               rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# T4: the oracle equals the page's composition of pad + grid_sample (fp64)

def page_composition(x, off, mask, p: Params):
    """dcnv3_core_pytorch's steps rebuilt from the walkthrough's description,
    with torch CPU binary64 library ops: pad, normalised reference points plus
    the dilation grid scaled by offset_scale, offset * offset_scale / extent,
    grid = 2*loc - 1, grid_sample(bilinear, zeros, align_corners=False), then
    the mask-weighted sum over points (softmax first for DCNv3)."""
    N, H, W, C = x.shape
    G, gc = p.G, p.gc
    xp = F.pad(x, [0, 0, p.pad_w, p.pad_w, p.pad_h, p.pad_h])
    Hin, Win = xp.shape[1], xp.shape[2]
    _, Ho, Wo, _, P, _ = off.shape
    ch = p.dilation_h * (p.kernel_h - 1) // 2
    cw = p.dilation_w * (p.kernel_w - 1) // 2
    ry = (ch + 0.5 + torch.arange(Ho, dtype=torch.float64) * p.stride_h) / Hin
    rx = (cw + 0.5 + torch.arange(Wo, dtype=torch.float64) * p.stride_w) / Win
    ref = torch.stack(torch.meshgrid(rx, ry, indexing="xy"), -1)           # (Ho, Wo, 2) as (x, y)
    gxs = [(ix * p.dilation_w - cw) / Win for ix in range(p.kernel_w)]
    gys = [(iy * p.dilation_h - ch) / Hin for iy in range(p.kernel_h)]
    pts = [(gx, gy) for ix, gx in enumerate(gxs) for iy, gy in enumerate(gys)
           if not (p.remove_center and ix == (p.kernel_w - 1) // 2 and iy == (p.kernel_h - 1) // 2)]
    grid = torch.tensor(pts, dtype=torch.float64)                          # (P, 2)
    norm = torch.tensor([Win, Hin], dtype=torch.float64)
    loc = ref[None, :, :, None, None, :] + grid * p.offset_scale + off * p.offset_scale / norm
    sgrid = 2 * loc - 1                                                    # (N, Ho, Wo, G, P, 2)
    planes = xp.reshape(N, Hin, Win, G, gc).permute(0, 3, 4, 1, 2).reshape(N * G, gc, Hin, Win)
    sgrid = sgrid.permute(0, 3, 1, 2, 4, 5).reshape(N * G, Ho * Wo, P, 2)
    s = F.grid_sample(planes, sgrid, mode="bilinear", padding_mode="zeros", align_corners=False)
    w = torch.softmax(mask, -1) if p.softmax else mask
    w = w.permute(0, 3, 1, 2, 4).reshape(N * G, 1, Ho * Wo, P)
    out = (s * w).sum(-1)                                                  # (N*G, gc, Ho*Wo)
    return out.reshape(N, G * gc, Ho, Wo).permute(0, 2, 3, 1)


T4_CASES = [
    dict(N=2, H=7, W=6, G=2, gc=3, softmax=1),
    dict(N=1, H=8, W=8, G=3, gc=2, softmax=0, stride_h=2, stride_w=2, dilation_h=2, dilation_w=2),
    dict(N=1, H=6, W=9, G=1, gc=4, softmax=1, remove_center=1, offset_scale=0.5),
    dict(N=2, H=5, W=5, G=2, gc=2, softmax=0, kernel_h=5, kernel_w=3, pad_h=2, pad_w=0),
    dict(N=1, H=9, W=7, G=2, gc=2, softmax=0, pad_h=3, pad_w=2, stride_w=3),
]


@pytest.mark.parametrize("case", T4_CASES)
def test_matches_grid_sample_composition(case):
    p = Params(**case)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(11)
    x = rng.uniform(-1, 1, (p.N, p.H, p.W, p.G * p.gc))
    off = rng.normal(0, 2, (p.N, ho, wo, p.G, P, 2))
    mask = rng.normal(0, 1, (p.N, ho, wo, p.G, P))
    go = rng.normal(0, 1, (p.N, ho, wo, p.G * p.gc))

    xt = torch.tensor(x, requires_grad=True)
    ot = torch.tensor(off, requires_grad=True)
    mt = torch.tensor(mask, requires_grad=True)
    ref = page_composition(xt, ot, mt, p)
    (ref * torch.tensor(go)).sum().backward()

    out = oracle.forward(p, x, off, mask)
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=0, atol=1e-12)
    gi, goff, gm = oracle.backward(p, go, x, off, mask)
    np.testing.assert_allclose(gi, xt.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(goff, ot.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(gm, mt.grad.numpy(), rtol=0, atol=1e-11)


# --------------------------------------------------------------------------
# T2: backward against central finite differences, and the adjoint identity

FD_CASES = [
    dict(softmax=0),
    dict(softmax=1),
    dict(softmax=0, stride_h=2, stride_w=2, dilation_h=2, dilation_w=2),
    dict(softmax=1, remove_center=1),
    dict(softmax=1, offset_scale=0.5),
]


def _off_knot_offsets(rng, shape, os):
    # fractional part of every sampling location kept in [0.15, 0.35] or
    # [0.65, 0.85] (taps may add a half pixel when offset_scale is 0.5), so a
    # small step never crosses a cell boundary.
    whole = rng.integers(-2, 3, shape).astype(np.float64)
    frac = rng.uniform(0.15, 0.35, shape)
    return (whole + frac) / os


@pytest.mark.parametrize("case", FD_CASES)
def test_backward_finite_differences(case):
    p = Params(N=1, H=5, W=5, G=2, gc=3, **case)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(12)
    x = rng.uniform(-1, 1, (1, 5, 5, 6))
    off = _off_knot_offsets(rng, (1, ho, wo, p.G, P, 2), p.offset_scale)
    mask = rng.normal(0, 1, (1, ho, wo, p.G, P))
    go = rng.normal(0, 1, (1, ho, wo, 6))
    gi, goff, gm = oracle.backward(p, go, x, off, mask)

    def loss(x_, off_, mask_):
        return float(np.sum(go * oracle.forward(p, x_, off_, mask_)))

    h = 1e-6
    for arr, grad in ((off, goff), (mask, gm), (x, gi)):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 60), replace=False)
        for i in idx:
            keep = flat[i]
            flat[i] = keep + h
            lp = loss(x, off, mask)
            flat[i] = keep - h
            lm = loss(x, off, mask)
            flat[i] = keep
            fd = (lp - lm) / (2 * h)
            assert abs(fd - gflat[i]) <= 1e-7 * (1 + abs(gflat[i])), (i, fd, gflat[i])


def test_grad_input_adjoint_identity():
    # the output is linear in the input: <go, J dx> == <J^T go, dx> exactly up to rounding
    p = Params(N=2, H=6, W=7, G=2, gc=3, softmax=1, stride_w=2)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(13)
    x = rng.uniform(-1, 1, (2, 6, 7, 6))
    dx = rng.uniform(-1, 1, x.shape)
    off = rng.normal(0, 2, (2, ho, wo, p.G, P, 2))
    mask = rng.normal(0, 1, (2, ho, wo, p.G, P))
    go = rng.normal(0, 1, (2, ho, wo, 6))
    gi, _, _ = oracle.backward(p, go, x, off, mask)
    lhs = np.sum(go * oracle.forward(p, dx, off, mask))
    assert abs(lhs - np.sum(gi * dx)) <= 1e-12 * max(1.0, abs(lhs))


# --------------------------------------------------------------------------
# the binary32 location mode equals the binary64 one wherever binary32 is exact

@pytest.mark.parametrize("softmax", [0, 1])
@pytest.mark.parametrize("os_", [1.0, 0.5])
def test_coord_f32_mode_matches_when_exact(softmax, os_):
    base = dict(N=1, H=7, W=8, G=2, gc=3, softmax=softmax, offset_scale=os_,
                stride_h=2, dilation_w=2, pad_w=2)
    p64, p32 = Params(**base), Params(coord_f32=1, **base)
    ho, wo, P = shapes(p64)
    rng = np.random.default_rng(14)
    x = rng.uniform(-1, 1, (1, 7, 8, 6))
    off = rng.integers(-512, 512, (1, ho, wo, 2, P, 2)) / 64.0   # exact in binary32
    mask = rng.normal(0, 1, (1, ho, wo, 2, P))
    go = rng.normal(0, 1, (1, ho, wo, 6))
    np.testing.assert_array_equal(oracle.forward(p32, x, off, mask), oracle.forward(p64, x, off, mask))
    for a, b in zip(oracle.backward(p32, go, x, off, mask), oracle.backward(p64, go, x, off, mask)):
        np.testing.assert_array_equal(a, b)


def test_coord_f32_mode_is_within_rounding_otherwise():
    p64 = Params(N=1, H=9, W=9, G=2, gc=3)
    p32 = Params(N=1, H=9, W=9, G=2, gc=3, coord_f32=1)
    ho, wo, P = shapes(p64)
    rng = np.random.default_rng(15)
    x = rng.uniform(-1, 1, (1, 9, 9, 6))
    off = rng.normal(0, 2, (1, ho, wo, 2, P, 2)).astype(np.float32).astype(np.float64)
    mask = rng.normal(0, 1, (1, ho, wo, 2, P))
    a, b = oracle.forward(p32, x, off, mask), oracle.forward(p64, x, off, mask)
    assert np.max(np.abs(a - b)) < 1e-5


# --------------------------------------------------------------------------
# the pixel-list entry points agree with the whole-tensor ones

def test_pixel_subsets_match_whole_tensor_results():
    p = Params(N=2, H=6, W=5, G=2, gc=3, softmax=1, stride_h=2)
    ho, wo, P = shapes(p)
    rng = np.random.default_rng(16)
    x = rng.uniform(-1, 1, (2, 6, 5, 6))
    off = rng.normal(0, 2, (2, ho, wo, 2, P, 2))
    mask = rng.normal(0, 1, (2, ho, wo, 2, P))
    go = rng.normal(0, 1, (2, ho, wo, 6))
    out = oracle.forward(p, x, off, mask)
    gi, goff, gm = oracle.backward(p, go, x, off, mask)
    allpix = np.arange(2 * ho * wo)
    np.testing.assert_array_equal(oracle.forward_pixels(p, x, off, mask, allpix),
                                  out.reshape(-1, 6))
    gi2, goff2, gm2 = oracle.backward_pixels(p, go, x, off, mask, allpix)
    np.testing.assert_allclose(gi2, gi, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(goff2, goff.reshape(-1, 2, P, 2))
    np.testing.assert_array_equal(gm2, gm.reshape(-1, 2, P))
    some = rng.choice(allpix, 7, replace=False)
    np.testing.assert_array_equal(oracle.forward_pixels(p, x, off, mask, some),
                                  out.reshape(-1, 6)[some])
    _, goff3, gm3 = oracle.backward_pixels(p, go, x, off, mask, some)
    np.testing.assert_array_equal(goff3, goff.reshape(-1, 2, P, 2)[some])
