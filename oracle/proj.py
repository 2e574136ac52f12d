"""The oracle of the linear projections around the core op.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark
may import it.  The product (the CUDA library and its binding) never imports,
links or calls it, and shares no code with it.

The DCN module surrounds the core op with dense linear layers.  DCNv3 (page
"没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三,
items 1-6) projects the input (input_proj), predicts the offsets and the mask
logits from the depthwise-convolved features with two linear layers, and
projects the core's output (output_proj).  DCNv4 merges the offset and mask
predictions into one linear layer (page "告别DCNv3的卡顿：实测DCNv4在A100上3倍提速，
手把手教你集成到FlashInternImage", section 1), whose output is the merged
offset/mask tensor the core op reads: per (pixel, group) a row of 2P offsets,
then P mask values, padded to the row stride.

Every one of those layers is y = x W^T + b over the rows of a channels-last
tensor, which is what this module computes, in binary64, with numpy's matrix
product as the one library step.

The centre feature scale (the InternImage-G walkthrough, section 三 item 5;
the DCNv4 guide, "高级配置参数详解") sits between the core and output_proj: a
sigmoid gate mixes the core's output with the centre pixel's own projected
feature x_proj.  The walkthrough gives the gate's function and inputs but not
its shape; this module takes one gate per (pixel, group), from G logits per
pixel (a linear layer of G outputs), applied to the group's gc channels:
    s = 1 / (1 + exp(-logit)),   out = core * (1 - s) + x_proj * s.
"""
from __future__ import annotations

import numpy as np


def linear(x, w, b=None) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * w[n, k] + b[n], in binary64.

    x: (M, K); w: (N, K), a linear layer's weight; b: (N,) or None."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"shapes {x.shape} and {w.shape} do not make x @ w.T")
    y = x @ w.T
    if b is not None:
        b = np.asarray(b, dtype=np.float64)
        if b.shape != (w.shape[0],):
            raise ValueError(f"bias shape {b.shape} for {w.shape[0]} outputs")
        y = y + b[None, :]
    return y


def merged_weights(w_offset, b_offset, w_mask, b_mask, G: int, P: int, row_stride: int):
    """The weight and bias of the merged offset/mask projection.

    w_offset: (G*P*2, K) and w_mask: (G*P, K), the two DCNv3-style layers whose
    outputs are the offset tensor (..., G, P, 2) and the mask tensor (..., G, P).
    Returns (w, b) of G*row_stride outputs: output g*row_stride + j is offset
    value j of group g for j < 2P, mask value j - 2P for 2P <= j < 3P, and zero
    (zero weights and bias) for the padding."""
    w_offset = np.asarray(w_offset, dtype=np.float64)
    w_mask = np.asarray(w_mask, dtype=np.float64)
    K = w_offset.shape[1]
    if w_offset.shape != (G * P * 2, K) or w_mask.shape != (G * P, K) or row_stride < 3 * P:
        raise ValueError("inconsistent merged-projection shapes")
    w = np.zeros((G * row_stride, K))
    b = np.zeros(G * row_stride)
    bo = np.zeros(G * P * 2) if b_offset is None else np.asarray(b_offset, dtype=np.float64)
    bm = np.zeros(G * P) if b_mask is None else np.asarray(b_mask, dtype=np.float64)
    for g in range(G):
        r = g * row_stride
        w[r:r + 2 * P] = w_offset[g * 2 * P:(g + 1) * 2 * P]
        b[r:r + 2 * P] = bo[g * 2 * P:(g + 1) * 2 * P]
        w[r + 2 * P:r + 3 * P] = w_mask[g * P:(g + 1) * P]
        b[r + 2 * P:r + 3 * P] = bm[g * P:(g + 1) * P]
    return w, b


def _gate(logits, M, G):
    l = np.asarray(logits, dtype=np.float64).reshape(M, G)
    with np.errstate(over="ignore"):  # exp(-l) = inf gives the limit s = 0
        return 1.0 / (1.0 + np.exp(-l))


def center_feature_scale(core, x_proj, logits, G: int) -> np.ndarray:
    """out[m, g*gc + c] = core * (1 - s[m, g]) + x_proj * s[m, g], with
    s = sigmoid(logits[m, g]), in binary64.

    core, x_proj: (M, C) rows of C = G * gc channels; logits: (M, G)."""
    core = np.asarray(core, dtype=np.float64)
    x = np.asarray(x_proj, dtype=np.float64)
    M, C = core.shape
    if x.shape != (M, C) or C % G:
        raise ValueError("inconsistent centre-feature-scale shapes")
    s = np.repeat(_gate(logits, M, G), C // G, axis=1)
    return core * (1.0 - s) + x * s


def center_feature_scale_backward(grad_out, core, x_proj, logits, G: int):
    """The gradients of center_feature_scale, in binary64:
    d core = g * (1 - s), d x_proj = g * s and
    d logit[m, k] = s (1 - s) * sum over group k's channels of g * (x_proj - core)
    (ds/dlogit = s (1 - s) for the logistic function).  Returns the three."""
    g = np.asarray(grad_out, dtype=np.float64)
    core = np.asarray(core, dtype=np.float64)
    x = np.asarray(x_proj, dtype=np.float64)
    M, C = core.shape
    s = _gate(logits, M, G)
    se = np.repeat(s, C // G, axis=1)
    dl = (g * (x - core)).reshape(M, G, C // G).sum(axis=2) * s * (1.0 - s)
    return g * (1.0 - se), g * se, dl
