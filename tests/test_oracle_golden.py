"""The oracle against hand-worked cases stored in tests/golden/hand_cases.json."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import Params

pytestmark = pytest.mark.usefixtures("oracle_lib")

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=[c["name"] for c in GOLDEN["cases"]])
@pytest.mark.parametrize("coord_f32", [0, 1])
def test_hand_case(case, coord_f32):
    p = Params(coord_f32=coord_f32, **case["params"])
    x, off, mask = (np.array(case[k], dtype=np.float64) for k in ("input", "offset", "mask"))
    tol = case["tol"]
    np.testing.assert_allclose(oracle.forward(p, x, off, mask), np.array(case["output"]),
                               rtol=0, atol=tol)
    gi, goff, gm = oracle.backward(p, np.array(case["grad_out"]), x, off, mask)
    for name, got in (("grad_input", gi), ("grad_offset", goff), ("grad_mask", gm)):
        if name in case:
            np.testing.assert_allclose(got, np.array(case[name]), rtol=0, atol=tol, err_msg=name)


@pytest.mark.parametrize("c", GOLDEN["out_shapes"]["cases"])
def test_out_shape(c):
    p = Params(N=1, H=c["H"], W=c["H"], G=1, gc=1, kernel_h=c["k"], kernel_w=c["k"],
               stride_h=c["stride"], stride_w=c["stride"], pad_h=c["pad"], pad_w=c["pad"],
               dilation_h=c["dilation"], dilation_w=c["dilation"])
    assert oracle.out_shape(p) == (c["H_out"], c["H_out"])


def test_workload_table_shapes_agree_with_oracle():
    from deformable_convolution_03_b300.inputs import WORKLOADS
    for w in WORKLOADS.values():
        p = Params(**w.params())
        assert oracle.out_shape(p) == (w.H_out, w.W_out), w.name
        assert oracle.num_points(p) == w.P == len(oracle.taps(p)), w.name
