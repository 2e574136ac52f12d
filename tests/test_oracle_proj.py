"""Pins of the projection oracle (oracle/proj.py) against values fixed by
hand and by the algebra of a linear layer, without a GPU."""
import json
import os

import numpy as np
import pytest

from oracle import proj

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "proj_cases.json")))


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=lambda c: "hand")
def test_hand_worked_case(case):
    y = proj.linear(case["x"], case["w"], case["b"])
    np.testing.assert_array_equal(y, np.array(case["y"], dtype=np.float64))


def test_identity_weight_copies_the_input():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 5))
    b = rng.standard_normal(5)
    np.testing.assert_array_equal(proj.linear(x, np.eye(5), None), x)
    np.testing.assert_array_equal(proj.linear(x, np.eye(5), b), x + b)


def test_one_hot_rows_select_input_columns():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 4))
    w = np.zeros((3, 4))
    w[0, 2] = 1.0
    w[1, 0] = 1.0
    w[2, 3] = 1.0
    np.testing.assert_array_equal(proj.linear(x, w), x[:, [2, 0, 3]])


def test_linear_in_input_and_weight():
    rng = np.random.default_rng(2)
    x1, x2 = rng.standard_normal((2, 9, 6))
    w1, w2 = rng.standard_normal((2, 4, 6))
    np.testing.assert_allclose(proj.linear(2 * x1 - 3 * x2, w1),
                               2 * proj.linear(x1, w1) - 3 * proj.linear(x2, w1), atol=1e-12)
    np.testing.assert_allclose(proj.linear(x1, 0.5 * w1 + w2),
                               0.5 * proj.linear(x1, w1) + proj.linear(x1, w2), atol=1e-12)


def test_output_columns_follow_weight_rows():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 6))
    w = rng.standard_normal((4, 6))
    perm = [2, 0, 3, 1]
    np.testing.assert_array_equal(proj.linear(x, w[perm]), proj.linear(x, w)[:, perm])


def test_shape_errors():
    with pytest.raises(ValueError):
        proj.linear(np.zeros((2, 3)), np.zeros((3, 2)))
    with pytest.raises(ValueError):
        proj.linear(np.zeros((2, 3)), np.zeros((4, 3)), np.zeros(3))


@pytest.mark.parametrize("G,P,rs", [(4, 9, 32), (2, 8, 24), (3, 9, 27)])
def test_merged_projection_splits_into_the_separate_ones(G, P, rs):
    # the merged layer's output, read as (M, G, rs), holds the offset layer's
    # output in [:2P], the mask layer's in [2P:3P] and zeros after
    rng = np.random.default_rng(4)
    M, K = 11, 16
    x = rng.standard_normal((M, K))
    wo, wm = rng.standard_normal((G * P * 2, K)), rng.standard_normal((G * P, K))
    bo, bm = rng.standard_normal(G * P * 2), rng.standard_normal(G * P)
    w, b = proj.merged_weights(wo, bo, wm, bm, G, P, rs)
    y = proj.linear(x, w, b).reshape(M, G, rs)
    np.testing.assert_allclose(y[:, :, :2 * P], proj.linear(x, wo, bo).reshape(M, G, 2 * P),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[:, :, 2 * P:3 * P], proj.linear(x, wm, bm).reshape(M, G, P),
                               rtol=0, atol=1e-12)
    assert np.all(y[:, :, 3 * P:] == 0)


# ---- the centre feature scale ------------------------------------------------

CFS = json.load(open(os.path.join(HERE, "golden", "cfs_cases.json")))


@pytest.mark.parametrize("case", CFS["cases"], ids=lambda c: f"G{c['G']}")
def test_centre_feature_scale_hand_worked(case):
    G = case["G"]
    out = proj.center_feature_scale(case["core"], case["x_proj"], case["logits"], G)
    np.testing.assert_allclose(out, case["out"], rtol=1e-14, atol=1e-14)
    gc, gx, gl = proj.center_feature_scale_backward(case["grad_out"], case["core"],
                                                    case["x_proj"], case["logits"], G)
    np.testing.assert_allclose(gc, case["grad_core"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(gx, case["grad_x_proj"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(gl, case["grad_logits"], rtol=1e-14, atol=1e-14)


def test_centre_feature_scale_saturated_and_even_gates():
    # a gate shut (s = 0) passes the core's output, an open one (s = 1) the
    # projected feature, s = 1/2 their mean
    rng = np.random.default_rng(5)
    core, x = rng.standard_normal((9, 12)), rng.standard_normal((9, 12))
    shut, open_, even = np.full((9, 3), -800.0), np.full((9, 3), 800.0), np.zeros((9, 3))
    np.testing.assert_array_equal(proj.center_feature_scale(core, x, shut, 3), core)
    np.testing.assert_array_equal(proj.center_feature_scale(core, x, open_, 3), x)
    np.testing.assert_allclose(proj.center_feature_scale(core, x, even, 3), (core + x) / 2,
                               rtol=1e-15, atol=1e-15)


def test_centre_feature_scale_gates_act_per_group():
    # moving group k's logit changes group k's channels and no other
    rng = np.random.default_rng(6)
    core, x = rng.standard_normal((4, 12)), rng.standard_normal((4, 12))
    l = rng.standard_normal((4, 3))
    base = proj.center_feature_scale(core, x, l, 3)
    for k in range(3):
        l2 = l.copy()
        l2[:, k] += 1.0
        d = proj.center_feature_scale(core, x, l2, 3) - base
        for j in range(3):
            moved = np.any(d[:, 4 * j:4 * j + 4] != 0)
            assert moved == (j == k)


def test_centre_feature_scale_backward_matches_finite_differences():
    # the derivative formulas against central differences of the forward,
    # for every input element of a small case
    rng = np.random.default_rng(7)
    M, G, gc = 3, 2, 3
    core, x = rng.standard_normal((M, G * gc)), rng.standard_normal((M, G * gc))
    l, g = rng.standard_normal((M, G)), rng.standard_normal((M, G * gc))
    gcore, gx, gl = proj.center_feature_scale_backward(g, core, x, l, G)
    h = 1e-6

    def loss(c, xx, ll):
        return float(np.sum(g * proj.center_feature_scale(c, xx, ll, G)))

    for arr, grad, which in ((core, gcore, 0), (x, gx, 1), (l, gl, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [core.copy(), x.copy(), l.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-7, atol=1e-8)
