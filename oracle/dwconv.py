"""The oracle of the offset branch's feature step: depthwise convolution,
LayerNorm and GELU.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark
may import it.  The product (the CUDA library and its binding) never imports,
links or calls it, and shares no code with it.

In the DCNv3 module the offsets and the mask are predicted from control
features x1, which a k x k depthwise convolution, LayerNorm and GELU extract
from the module's input (page
"没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三
item 2; the page's configuration table gives dw_kernel_size 5).  The page
names the three steps and the kernel size only.  This module takes the
plainest reading of each:

  * depthwise convolution: every channel c convolved with its own k x k
    kernel, stride 1, zero padding (k - 1) / 2 (the output has the input's
    size, one feature vector per pixel, as the projections that follow need),
    plus a per-channel bias; a convolution layer's cross-correlation:
        y[n, i, j, c] = b[c] + sum_{a, e} w[a, e, c] * x[n, i + a - r, j + e - r, c]
    with r = (k - 1) / 2 and x zero outside the image;
  * LayerNorm over the C channels of each pixel, biased variance, eps given:
        z = (y - mean) / sqrt(var + eps) * gamma + beta;
  * GELU in its exact form: g(z) = z / 2 * (1 + erf(z / sqrt(2))).

Everything is binary64; math.erf is the one library step.  Tensors are
channels-last: x (N, H, W, C), w (k, k, C), b, gamma, beta (C,).
"""
from __future__ import annotations

import math

import numpy as np


def dwconv(x, w, b) -> np.ndarray:
    """The depthwise convolution with zero padding (k - 1) / 2, binary64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    N, H, W, C = x.shape
    k = w.shape[0]
    if w.shape != (k, k, C) or k % 2 == 0 or b.shape != (C,):
        raise ValueError(f"kernel {w.shape} / bias {b.shape} for {C} channels")
    r = (k - 1) // 2
    xp = np.zeros((N, H + 2 * r, W + 2 * r, C))
    xp[:, r:r + H, r:r + W, :] = x
    y = np.zeros((N, H, W, C))
    for a in range(k):          # kernel row: input row i + a - r
        for e in range(k):      # kernel column: input column j + e - r
            y += w[a, e][None, None, None, :] * xp[:, a:a + H, e:e + W, :]
    return y + b[None, None, None, :]


def layer_norm(y, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm over the last (channel) axis, biased variance, binary64."""
    y = np.asarray(y, dtype=np.float64)
    mean = y.mean(axis=-1, keepdims=True)
    var = ((y - mean) ** 2).mean(axis=-1, keepdims=True)
    return (y - mean) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + \
        np.asarray(beta, np.float64)


def gelu(z) -> np.ndarray:
    """z / 2 * (1 + erf(z / sqrt(2))), binary64."""
    z = np.asarray(z, dtype=np.float64)
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def dwconv_ln_gelu(x, w, b, gamma, beta, eps: float) -> np.ndarray:
    """x1 = GELU(LayerNorm(dwconv(x))), the offset branch's control features."""
    return gelu(layer_norm(dwconv(x, w, b), gamma, beta, eps))
