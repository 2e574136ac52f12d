"""dcn_core_bwd_noalloc: the backward for callers that cannot allocate.

Some callers may not allocate device memory where they run the backward (a
plugin inside a runtime that owns all device memory, or code with a fixed
memory budget), so they cannot hand dcn_core_bwd the float32 workspace that
float16 / bfloat16 need.  dcn_core_bwd_noalloc takes that accumulator from a
static array inside the library instead.  These tests check its results
against the oracle and against dcn_core_bwd, on two calls in a row (the array
keeps the previous call's contents, which must not leak into the next
result), and that requests larger than the array are refused before any
CUDA call.

This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import WORKLOADS, make_inputs

import oracle
from parity import assert_close, f64, lib_params, oracle_params


def _backward(w, t, noalloc: bool):
    p = lib_params(w)
    g, i, o, m = (t[k].cuda() for k in ("grad_out", "input", "offset", "mask"))
    gi, go, gm = torch.empty_like(i), torch.empty_like(o), torch.empty_like(m)
    if noalloc:
        rc = B.lib().dcn_core_bwd_noalloc(ctypes.byref(p.c()), g.data_ptr(), i.data_ptr(),
                                          o.data_ptr(), m.data_ptr(), gi.data_ptr(),
                                          go.data_ptr(), gm.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
        assert rc == B.DCN_OK, B.dcn_status_str(rc)
    else:
        nbytes = B.dcn_core_bwd_workspace(p)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        B.dcn_core_bwd(p, g, i, o, m, gi, go, gm, ws, nbytes)
    torch.cuda.synchronize()
    return gi, go, gm


@pytest.mark.gpu
@pytest.mark.usefixtures("native", "oracle_lib")
@pytest.mark.parametrize("name", ["t_stage1_f16", "g_stage1_rc_bf16", "fb28_f32"])
def test_noalloc_backward_matches_oracle_and_workspace_backward(name):
    base = WORKLOADS[name]
    w = base.with_(N=8 if base.N > 8 else base.N, backward=True)
    if base.name.startswith("g_stage1"):
        w = base.with_(N=1, H=64, W=64, H_out=64, W_out=64, backward=True)
    assert B.dcn_core_bwd_workspace(lib_params(w)) <= B.DCN_NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((11, 12)):   # two calls in a row share the array
        t = make_inputs(w, seed=seed, grad=True)
        want = _backward(w, t, noalloc=False)
        got = _backward(w, t, noalloc=True)
        ref = oracle.backward(oracle_params(w), f64(t["grad_out"]), f64(t["input"]),
                              f64(t["offset"]), f64(t["mask"]))
        for name_, a, b, r in zip(("grad_input", "grad_offset", "grad_mask"), got, want, ref):
            assert_close(a, r, w.dtype, f"call {call}: {name_} against the oracle")
            assert_close(a, f64(b), w.dtype, f"call {call}: {name_} against dcn_core_bwd")


@pytest.mark.usefixtures("native")
def test_noalloc_refuses_requests_beyond_the_scratch():
    # 64 images of 56x56x64 need 51 MB of accumulator: refused before any CUDA
    # call.  The tensors are NULL: the size check comes before the pointer
    # check, and a call that got past it would stop at DCN_ERR_NULL, never
    # at a launch.
    w = WORKLOADS["t_stage1_f16"]
    p = lib_params(w)
    assert B.dcn_core_bwd_workspace(p) > B.DCN_NOALLOC_SCRATCH_BYTES
    rc = B.lib().dcn_core_bwd_noalloc(ctypes.byref(p.c()), None, None, None, None, None, None,
                                      None, None)
    assert rc == B.DCN_ERR_UNSUPPORTED
    bad = lib_params(w.with_(N=-1))
    assert B.lib().dcn_core_bwd_noalloc(ctypes.byref(bad.c()), None, None, None, None, None,
                                        None, None, None) == B.DCN_ERR_SHAPE
