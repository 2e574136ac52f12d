"""DCNv4's merged offset/mask layout (dcn_core_fwd_om / dcn_core_bwd_om)
against the oracle, which takes the same values as separate tensors."""
import numpy as np
import pytest
import torch

import oracle
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import WORKLOADS, Workload, make_inputs
from parity import assert_close, f64, lib_params, oracle_params

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native", "oracle_lib")]


def merged(offset: torch.Tensor, mask: torch.Tensor, stride: int) -> torch.Tensor:
    """(N,Ho,Wo,G,stride): 2P offsets, P mask values, NaN padding."""
    N, Ho, Wo, G, P, _ = offset.shape
    pad = torch.full((N, Ho, Wo, G, stride - 3 * P), float("nan"), dtype=offset.dtype)
    return torch.cat([offset.reshape(N, Ho, Wo, G, 2 * P), mask, pad], dim=-1).contiguous()


CASES = [
    ("t_stage1_f16", dict(), 32),
    ("g_stage1_rc_bf16", dict(N=1), 24),
    ("fb28_f32", dict(N=8), 28),
    ("fb28_s2d2_f32", dict(N=8), 30),
    ("v3_tiny_f32", dict(), 28),
]


BWD = {
    "default": {},
    "split": {"bwd_split": 1},
    "single_pass": {"bwd_split": 0},
}


@pytest.mark.parametrize("bwd", list(BWD))
@pytest.mark.parametrize("name,over,stride", CASES, ids=[c[0] for c in CASES])
def test_merged_layout_forward_and_backward(name, over, stride, bwd, opts):
    # every backward path reads the merged rows and writes their padding
    opts.update(BWD[bwd])
    w = WORKLOADS[name].with_(backward=True, **over)
    t = make_inputs(w, grad=True)
    p = lib_params(w)
    dev = "cuda"
    om = merged(t["offset"], t["mask"], stride).to(dev)
    x, go = t["input"].to(dev), t["grad_out"].to(dev)
    out = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=x.dtype, device=dev)
    B.dcn_core_fwd_om(p, x, om, stride, out)
    gi = torch.empty_like(x)
    gom = torch.full_like(om, float("nan"))
    nbytes = B.dcn_core_bwd_workspace(p)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    B.dcn_core_bwd_om(p, go, x, om, stride, gi, gom, ws, nbytes)
    torch.cuda.synchronize()

    q = oracle_params(w)
    f = {k: f64(v) for k, v in t.items()}
    assert_close(out, oracle.forward(q, f["input"], f["offset"], f["mask"]), w.dtype, "output")
    rgi, rgo, rgm = oracle.backward(q, f["grad_out"], f["input"], f["offset"], f["mask"])
    P = w.P
    assert_close(gi, rgi, w.dtype, "grad_input")
    assert_close(gom[..., :2 * P].reshape(rgo.shape), rgo, w.dtype, "grad_offset")
    assert_close(gom[..., 2 * P:3 * P], rgm, w.dtype, "grad_mask")
    assert torch.all(gom[..., 3 * P:] == 0), "padding of grad_offset_mask"


def test_merged_equals_separate_bitwise():
    # the same kernels read the same values: identical forward results
    w = WORKLOADS["t_stage2_bf16"].with_(N=4)
    t = make_inputs(w)
    p = lib_params(w)
    x, o, m = (t[k].cuda() for k in ("input", "offset", "mask"))
    a = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=x.dtype, device="cuda")
    b = torch.empty_like(a)
    B.dcn_core_fwd(p, x, o, m, a)
    B.dcn_core_fwd_om(p, x, merged(t["offset"], t["mask"], 32).cuda(), 32, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
