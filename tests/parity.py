"""Helpers of the GPU parity tests: run the CUDA library and the oracle on the
same seeded inputs and compare under the stated tolerances.

Tolerances (applied separately to output, grad_input, grad_offset, grad_mask):
  float32:            max|gpu - ref| <= 1e-4  and  max|gpu - ref| <= 1e-5 * max|ref|
  float16 / bfloat16: max|gpu - ref| <= 2e-2 * max|ref|
The reference is the binary64 oracle evaluated on the very values the GPU
receives (16-bit inputs upcast exactly), with the sampling location formed in
binary32 like the kernels form it, so that both sides take floor() of the same
number.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import DTYPES, Workload


def oracle_params(w: Workload) -> oracle.Params:
    return oracle.Params(coord_f32=1, **w.params())


def lib_params(w: Workload) -> B.Params:
    return B.Params(dtype=B.TORCH_TO_DCN[DTYPES[w.dtype]], **w.params())


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got: torch.Tensor, ref: np.ndarray) -> tuple[float, float]:
    g = f64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite values"
    return float(np.max(np.abs(g - ref))) if g.size else 0.0, \
        float(np.max(np.abs(ref))) if ref.size else 0.0


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str) -> None:
    err, mx = errors(got, ref)
    if dtype == "f32":
        assert err <= 1e-4 and err <= 1e-5 * mx, f"{what}: max err {err:.3e}, max|ref| {mx:.3e}"
    else:
        assert err <= 2e-2 * mx, f"{what}: max err {err:.3e} > 2e-2 * {mx:.3e}"


def run_fwd(w: Workload, t: dict, dev="cuda") -> torch.Tensor:
    p = lib_params(w)
    i, o, m = (t[k].to(dev).contiguous() for k in ("input", "offset", "mask"))
    out = torch.full((w.N, w.H_out, w.W_out, w.C), float("nan"), dtype=i.dtype, device=dev)
    B.dcn_core_fwd(p, i, o, m, out)
    torch.cuda.synchronize()
    return out


def run_bwd(w: Workload, t: dict, dev="cuda"):
    p = lib_params(w)
    g, i, o, m = (t[k].to(dev).contiguous() for k in ("grad_out", "input", "offset", "mask"))
    gi = torch.full_like(i, float("nan"))
    go = torch.full_like(o, float("nan"))
    gm = torch.full_like(m, float("nan"))
    nbytes = B.dcn_core_bwd_workspace(p)
    ws = torch.full((max(nbytes // 4, 1),), float("nan"), device=dev) if nbytes else None
    B.dcn_core_bwd(p, g, i, o, m, gi, go, gm, ws, nbytes)
    torch.cuda.synchronize()
    return gi, go, gm


def check_fwd(w: Workload, t: dict) -> None:
    out = run_fwd(w, t)
    ref = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    assert_close(out, ref, w.dtype, f"{w.name} output")


def check_bwd(w: Workload, t: dict) -> None:
    gi, go, gm = run_bwd(w, t)
    rgi, rgo, rgm = oracle.backward(oracle_params(w), f64(t["grad_out"]), f64(t["input"]),
                                    f64(t["offset"]), f64(t["mask"]))
    assert_close(gi, rgi, w.dtype, f"{w.name} grad_input")
    assert_close(go, rgo, w.dtype, f"{w.name} grad_offset")
    assert_close(gm, rgm, w.dtype, f"{w.name} grad_mask")
