"""Pins of the oracle's offset-branch feature step (oracle/dwconv.py):
depthwise convolution, LayerNorm and GELU, each pinned apart from the oracle's
own code: against torch's binary64 conv2d / layer_norm / gelu (independent
library implementations of the same definitions), hand-worked values, exact
special cases and identities.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dwconv as D

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "dwconv_cases.json")))


def rand(shape, seed):
    return np.random.default_rng(seed).uniform(-1, 1, shape)


def torch_ref(x, w, b, gamma, beta, eps):
    """torch binary64: conv2d with groups = C (cross-correlation), layer_norm, gelu."""
    C, k = x.shape[-1], w.shape[0]
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1)          # (C, 1, k, k)
    y = F.conv2d(xt, wt, torch.from_numpy(b), padding=(k - 1) // 2, groups=C)
    y = y.permute(0, 2, 3, 1)
    z = F.layer_norm(y, (C,), torch.from_numpy(gamma), torch.from_numpy(beta), eps)
    return y.numpy(), z.numpy(), F.gelu(z).numpy()


@pytest.mark.parametrize("N,H,W,C,k", [(1, 6, 7, 1, 3), (2, 5, 9, 5, 5), (1, 3, 4, 64, 5),
                                       (2, 8, 8, 16, 7), (1, 4, 3, 8, 1), (1, 2, 11, 3, 5)])
@pytest.mark.parametrize("eps", [1e-5, 1e-6])
def test_matches_torch_binary64(N, H, W, C, k, eps):
    x = rand((N, H, W, C), 1)
    w, b = rand((k, k, C), 2), rand((C,), 3)
    gamma, beta = 1 + 0.5 * rand((C,), 4), rand((C,), 5)
    y_ref, z_ref, g_ref = torch_ref(x, w, b, gamma, beta, eps)
    np.testing.assert_allclose(D.dwconv(x, w, b), y_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(D.layer_norm(y_ref, gamma, beta, eps), z_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(D.gelu(z_ref), g_ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(D.dwconv_ln_gelu(x, w, b, gamma, beta, eps), g_ref, rtol=0,
                               atol=1e-12)


@pytest.mark.parametrize("k", [3, 5])
def test_delta_input_reproduces_the_flipped_kernel(k):
    # a cross-correlation: one nonzero input at (i0, j0) appears at output
    # (i0 - a + r, j0 - e + r) with weight w[a, e]; other channels stay zero
    r = (k - 1) // 2
    H, W, C, c = 9, 8, 3, 1
    w = rand((k, k, C), 7)
    for i0, j0 in ((4, 3), (0, 0), (8, 7), (1, 6)):
        x = np.zeros((1, H, W, C))
        x[0, i0, j0, c] = 1.0
        y = D.dwconv(x, w, np.zeros(C))
        want = np.zeros((1, H, W, C))
        for a in range(k):
            for e in range(k):
                i, j = i0 - a + r, j0 - e + r
                if 0 <= i < H and 0 <= j < W:
                    want[0, i, j, c] = w[a, e, c]
        np.testing.assert_array_equal(y, want)


def test_constant_input_counts_the_taps_inside_the_image():
    # zero padding: a ones kernel on a ones image counts the in-image taps
    H, W, k = 6, 7, 5
    y = D.dwconv(np.ones((1, H, W, 1)), np.ones((k, k, 1)), np.zeros(1))[0, :, :, 0]
    r = 2
    rows = np.array([min(i + r, H - 1) - max(i - r, 0) + 1 for i in range(H)])
    cols = np.array([min(j + r, W - 1) - max(j - r, 0) + 1 for j in range(W)])
    np.testing.assert_array_equal(y, np.outer(rows, cols).astype(float))


def test_bias_adds_per_channel():
    x, w = rand((1, 4, 4, 3), 9), rand((3, 3, 3), 10)
    b = np.array([0.5, -2.0, 7.0])
    np.testing.assert_allclose(D.dwconv(x, w, b) - D.dwconv(x, w, np.zeros(3)),
                               np.broadcast_to(b, (1, 4, 4, 3)), rtol=0, atol=1e-14)


def test_layer_norm_identities():
    # gamma 1, beta 0: per pixel the normalised values have mean 0 and mean
    # square var / (var + eps); gamma and beta then act affinely per channel
    y = rand((2, 3, 4, 10), 11) * 5
    eps = 1e-5
    z = D.layer_norm(y, np.ones(10), np.zeros(10), eps)
    var = y.var(axis=-1)
    np.testing.assert_allclose(z.mean(axis=-1), 0, atol=1e-14)
    np.testing.assert_allclose((z ** 2).mean(axis=-1), var / (var + eps), rtol=1e-13)
    g, bt = rand((10,), 12), rand((10,), 13)
    np.testing.assert_allclose(D.layer_norm(y, g, bt, eps), z * g + bt, rtol=0, atol=1e-13)
    # a constant pixel normalises to beta
    np.testing.assert_allclose(D.layer_norm(np.full((1, 1, 1, 10), 3.0), g, bt, eps)[0, 0, 0], bt,
                               atol=1e-15)


def test_gelu_values():
    gv = GOLDEN["gelu_values"]
    np.testing.assert_allclose(D.gelu(np.array(gv["z"])), np.array(gv["gelu"]), rtol=0,
                               atol=1e-15)
    # far from zero GELU is the identity above and zero below
    np.testing.assert_allclose(D.gelu(np.array([40.0, -40.0])), [40.0, 0.0], atol=1e-300)


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=[c["name"] for c in GOLDEN["cases"]])
def test_hand_case(case):
    H, W, k, eps = case["H"], case["W"], case["k"], case["eps"]
    w = np.zeros((k, k, 2))
    w[..., 0], w[..., 1] = 1.0, 2.0
    out = D.dwconv_ln_gelu(np.ones((1, H, W, 2)), w, np.zeros(2), np.ones(2), np.zeros(2), eps)
    t = np.array(case["taps"], dtype=float)
    np.testing.assert_array_equal(D.dwconv(np.ones((1, H, W, 2)), w, np.zeros(2))[0, :, :, 0], t)
    zz = 0.5 * t / np.sqrt(0.25 * t * t + eps)            # (-zz, +zz) per pixel
    phi = lambda v: 0.5 * (1 + np.vectorize(math.erf)(v / math.sqrt(2)))   # normal CDF
    np.testing.assert_allclose(out[0, :, :, 0], -zz * phi(-zz), rtol=1e-14)
    np.testing.assert_allclose(out[0, :, :, 1], zz * phi(zz), rtol=1e-14)
