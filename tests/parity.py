"""Helpers of the GPU parity tests: run the CUDA library and the oracle on the
same seeded inputs and compare under the stated tolerances.

Tolerances (applied separately to output, grad_input, grad_offset, grad_mask):
  float32:            max|gpu - ref| <= 1e-4  and  max|gpu - ref| <= 1e-5 * max|ref|
  float16 / bfloat16: max|gpu - ref| <= 2e-2 * max|ref|
The reference is the binary64 oracle evaluated on the very values the GPU
receives (16-bit inputs upcast exactly), with the sampling location formed in
binary32 like the kernels form it, so that both sides take floor() of the same
number.

Every buffer the library writes (outputs and the workspace) is the middle of a
larger allocation whose guard regions before and after hold a canary pattern;
after each call the guards must be untouched, so that a write outside a
tensor shows up as a failure here (the mechanical bounds check that stands in
for a memory checker).
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


# Guard elements on each side of a written buffer: 256 bytes of any dtype, so
# the buffer keeps the allocation's alignment.
GUARD_BYTES = 256
CANARY = -768.0   # exact in float32, float16 and bfloat16


class Guarded:
    """A device tensor of `shape` (filled with NaN) inside a larger allocation
    whose guard regions hold CANARY."""

    def __init__(self, shape, dtype, dev="cuda"):
        es = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // es
        n = 1
        for d in shape:
            n *= d
        self.flat = torch.full((n + 2 * self.g,), CANARY, dtype=dtype, device=dev)
        self.t = self.flat[self.g:self.g + n].view(shape)
        self.t.fill_(float("nan"))

    def check(self, what: str) -> None:
        for part in (self.flat[:self.g], self.flat[self.flat.numel() - self.g:]):
            assert bool(torch.all(part == CANARY)), f"{what}: a guard region was overwritten"


def run_fwd(w: Workload, t: dict, dev="cuda") -> torch.Tensor:
    p = lib_params(w)
    i, o, m = (t[k].to(dev).contiguous() for k in ("input", "offset", "mask"))
    out = Guarded((w.N, w.H_out, w.W_out, w.C), i.dtype, dev)
    B.dcn_core_fwd(p, i, o, m, out.t)
    torch.cuda.synchronize()
    out.check(f"{w.name} output")
    return out.t


def run_bwd(w: Workload, t: dict, dev="cuda"):
    p = lib_params(w)
    g, i, o, m = (t[k].to(dev).contiguous() for k in ("grad_out", "input", "offset", "mask"))
    gi, go, gm = (Guarded(x.shape, x.dtype, dev) for x in (i, o, m))
    nbytes = B.dcn_core_bwd_workspace(p)
    ws = Guarded((max(nbytes // 4, 1),), torch.float32, dev) if nbytes else None
    B.dcn_core_bwd(p, g, i, o, m, gi.t, go.t, gm.t, ws.t if ws else None, nbytes)
    torch.cuda.synchronize()
    for name, b in (("grad_input", gi), ("grad_offset", go), ("grad_mask", gm),
                    ("workspace", ws)):
        if b is not None:
            b.check(f"{w.name} {name}")
    return gi.t, go.t, gm.t


def check_fwd(w: Workload, t: dict, coord_f32: int = 1) -> None:
    """The forward against the oracle.  coord_f32=0 evaluates the oracle with
    its locations in binary64 throughout: the forward's output is continuous
    across cell edges, so it must pass the same tolerance without sharing the
    kernels' binary32 location."""
    out = run_fwd(w, t)
    q = oracle_params(w)
    q.coord_f32 = coord_f32
    ref = oracle.forward(q, f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    assert_close(out, ref, w.dtype, f"{w.name} output")


def check_bwd(w: Workload, t: dict) -> None:
    gi, go, gm = run_bwd(w, t)
    rgi, rgo, rgm = oracle.backward(oracle_params(w), f64(t["grad_out"]), f64(t["input"]),
                                    f64(t["offset"]), f64(t["mask"]))
    assert_close(gi, rgi, w.dtype, f"{w.name} grad_input")
    assert_close(go, rgo, w.dtype, f"{w.name} grad_offset")
    assert_close(gm, rgm, w.dtype, f"{w.name} grad_mask")
