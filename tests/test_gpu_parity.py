"""GPU parity: the CUDA library against the oracle, element by element.

Full-size runs of every workload (the five configurations), small ragged
cases over dtypes / group widths / geometries / kernel instances, and the
degenerate cases (exact copies, samples out of the image, empty batch,
misaligned slices, non-default streams, more than 2^31 input elements).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from deformable_convolution_03_b300 import binding as B
from deformable_convolution_03_b300.inputs import SUITES, WORKLOADS, Workload, make_inputs
from parity import (assert_close, check_bwd, check_fwd, f64, lib_params, oracle_params, run_bwd,
                    run_fwd)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("native", "oracle_lib")]

HERE = os.path.dirname(os.path.abspath(__file__))


def small(name, dtype="f32", **kw) -> Workload:
    """A small workload; output size and point count taken from the oracle."""
    base = dict(N=2, H=9, W=7, G=2, gc=8, offset_std=2.0, seed=77)
    base.update(kw)
    q = oracle.Params(**{k: v for k, v in base.items() if k in oracle.Params.__dataclass_fields__})
    ho, wo = oracle.out_shape(q)
    return Workload(name=name, dtype=dtype, H_out=ho, W_out=wo, P=oracle.num_points(q),
                    backward=True, **base)


# ---- the five configurations at full size -------------------------------------

ALL = [n for suite in SUITES.values() for n in suite]


@pytest.mark.parametrize("name", ALL)
def test_config_forward_full_size(name):
    w = WORKLOADS[name]
    check_fwd(w, make_inputs(w))


@pytest.mark.parametrize("name", SUITES["dcnv4_fwd_bwd_f32"])
def test_config_backward_full_size(name):
    w = WORKLOADS[name]
    check_bwd(w, make_inputs(w))


BWD16 = SUITES["dcnv4_t_stage1_f16"] + SUITES["dcnv4_t_stages_bf16"] + SUITES["dcnv3_g_stage1_bf16"]


@pytest.mark.parametrize("name", BWD16)
def test_config_backward_16bit_full_size(name):
    # the 16-bit backward at the full size the benchmark times (64 images at
    # the FlashInternImage-T stages, InternImage-G stage 1 with and without
    # its centre tap), every element against the oracle
    w = WORKLOADS[name].with_(backward=True)
    check_bwd(w, make_inputs(w, grad=True))


@pytest.mark.parametrize("name", BWD16)
def test_config_forward_against_binary64_locations(name):
    # the oracle with its sampling locations in binary64 throughout (no shared
    # binary32 rounding before floor): the forward is continuous across cell
    # edges, so it must meet the same tolerance
    w = WORKLOADS[name]
    check_fwd(w, make_inputs(w), coord_f32=0)


# ---- small ragged cases --------------------------------------------------------

RAGGED = []
for dt in ("f32", "f16", "bf16"):
    for gc in (1, 3, 5, 8, 12, 16, 24, 32, 48, 64):
        for sm in (0, 1):
            RAGGED.append(small(f"{dt}_gc{gc}_sm{sm}", dt, gc=gc, softmax=sm, G=3 if gc < 8 else 2))

GEOMS = [
    small("s2", stride_h=2, stride_w=2),
    small("s2d2", stride_h=2, stride_w=2, dilation_h=2, dilation_w=2, H=28, W=28),
    small("k5x3", kernel_h=5, kernel_w=3, pad_h=2, pad_w=0, stride_w=2),
    small("k1", kernel_h=1, kernel_w=1, pad_h=0, pad_w=0),
    small("k7rc", kernel_h=7, kernel_w=7, pad_h=3, pad_w=3, remove_center=1, H=12, W=11,
          softmax=1),
    small("k8x8", kernel_h=8, kernel_w=8, pad_h=3, pad_w=4, H=12, W=13, gc=4),   # P = 64
    small("os_half", offset_scale=0.5, softmax=1),
    small("nopad_d3", pad_h=0, pad_w=3, dilation_w=3),
    small("wide_off", offset_std=6.0),
    small("one_px", H=1, W=1, N=3, gc=16),
    small("big_gc", G=1, gc=512, H=5, W=6, N=1),
]


@pytest.mark.parametrize("w", RAGGED + GEOMS, ids=lambda w: w.name)
def test_small_forward_and_backward(w):
    t = make_inputs(w)
    check_fwd(w, t)
    check_bwd(w, t)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cap", [1, 2, 4, 8, 16, 32])
def test_every_general_kernel_instance(dt, cap, opts):
    # force each channels-per-thread instance of the general kernels
    opts.update({"fwd_wide": 0, "bwd_split": 0,
                 "fwd_cpt": cap, "bwd_cpt": cap})
    w = small(f"inst_{dt}_{cap}", dt, gc=32, G=2, softmax=1, N=3, H=10, W=9)
    t = make_inputs(w)
    check_fwd(w, t)
    check_bwd(w, t)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("gc", [4, 8, 16, 24, 48])
@pytest.mark.parametrize("sm,rc", [(0, 0), (1, 0), (1, 1)])
@pytest.mark.parametrize("tile", ["1", "0"])
def test_wide_forward_instances(dt, gc, sm, rc, tile, opts):
    # slices of 4, 8 and 16 channels, 9 points and the runtime point count,
    # blocks over 2-D pixel tiles and over consecutive items
    opts.update({"fwd_tma": 0, "fwd_tile": int(tile)})
    w = small(f"wide_{dt}_{gc}", dt, gc=gc, G=3, softmax=sm, remove_center=rc, N=2, H=11, W=13)
    check_fwd(w, make_inputs(w))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("gc,G", [(8, 4), (16, 4), (16, 8), (32, 4), (48, 2)])
@pytest.mark.parametrize("sm,rc", [(0, 0), (1, 0), (1, 1)])
@pytest.mark.parametrize("halo", ["6", "2", "0"])
def test_tma_forward_instances(dt, gc, G, sm, rc, halo, opts):
    # the forward with its input window staged by a tensor copy: every slice
    # width, one or several blocks per tile's groups (a pixel's channels over
    # 128 bytes), the 9-point, 8-point and runtime instances; halos of 6, 2
    # and 0 pixels send more and more samples through the far path
    opts.set("fwd_halo", int(halo))
    w = small(f"tma_{dt}_{gc}_{G}", dt, gc=gc, G=G, softmax=sm, remove_center=rc, N=2, H=19,
              W=21, offset_std=3.0)
    check_fwd(w, make_inputs(w))


@pytest.mark.parametrize("k", [5, 7])
@pytest.mark.parametrize("win_kb", [64, 112])
def test_large_kernels_window_budget(k, win_kb, opts):
    # 5 x 5 and 7 x 7 taps at FlashInternImage-T stage 1's plane (4 images):
    # with 64 KB a 7 x 7 window keeps a halo of 3 and takes up to 112 KB
    # instead; both budgets against the oracle, offsets N(0, 2)
    opts.set("fwd_big_win", win_kb)
    w = WORKLOADS["t_stage1_f16"].with_(name=f"t1_k{k}_{win_kb}", N=4, kernel_h=k, kernel_w=k,
                                        pad_h=k // 2, pad_w=k // 2, P=k * k)
    check_fwd(w, make_inputs(w))


@pytest.mark.parametrize("geom", ["s2d2", "k5", "k7rc", "k1"])
def test_tma_forward_geometries(geom):
    # windows for strided, dilated and larger kernels, and for 1x1
    over = {"s2d2": dict(stride_h=2, stride_w=2, dilation_h=2, dilation_w=2),
            "k5": dict(kernel_h=5, kernel_w=5, pad_h=2, pad_w=2, offset_scale=0.5),
            "k7rc": dict(kernel_h=7, kernel_w=7, pad_h=3, pad_w=3, remove_center=1),
            "k1": dict(kernel_h=1, kernel_w=1, pad_h=0, pad_w=0)}[geom]
    w = small(f"tmag_{geom}", "bf16", gc=16, G=4, N=2, H=23, W=26, **over)
    check_fwd(w, make_inputs(w))


@pytest.mark.parametrize("H,W", [(14, 14), (7, 7), (13, 9), (5, 30), (30, 5), (1, 40), (40, 1),
                                 (3, 3)])
@pytest.mark.parametrize("dt,gc,G", [("f16", 16, 4), ("bf16", 16, 16), ("bf16", 32, 2)])
def test_tma_forward_plane_shapes(H, W, dt, gc, G):
    # small and elongated planes, where the tile of fewest warps is not a
    # power of two (7 x 7, 14 x 4, 1 x 40 ...) and blocks have fewer than 256
    # threads
    w = small(f"tmap_{dt}_{gc}_{G}_{H}x{W}", dt, gc=gc, G=G, N=3, H=H, W=W, offset_std=2.0)
    check_fwd(w, make_inputs(w))


SPLIT = [
    small("sp_f16_g16", "f16", gc=16, G=4, N=2, H=21, W=19),
    small("sp_f32_far", "f32", gc=16, G=2, N=2, H=20, W=23, offset_std=7.0),
    small("sp_bf16_s2d2", "bf16", gc=16, G=2, N=2, H=28, W=27, stride_h=2, stride_w=2,
          dilation_h=2, dilation_w=2, softmax=1),
    small("sp_f16_g8", "f16", gc=8, G=5, N=1, H=17, W=33),
    small("sp_f32_g4", "f32", gc=4, G=3, N=2, H=9, W=40, softmax=1),
    small("sp_bf16_g32", "bf16", gc=32, G=2, N=1, H=35, W=18, remove_center=1, softmax=1),
    small("sp_f32_g64", "f32", gc=64, G=1, N=2, H=13, W=11),
    small("sp_f16_g128", "f16", gc=128, G=2, N=1, H=9, W=10),
    small("sp_f32_k5neg", "f32", gc=8, G=2, N=1, H=16, W=16, kernel_h=5, kernel_w=5, pad_h=2,
          pad_w=2, offset_scale=-0.75),
    small("sp_f16_1px", "f16", gc=16, G=2, N=3, H=1, W=1),
    small("sp_f32_s3", "f32", gc=16, G=1, N=1, H=37, W=41, stride_h=3, stride_w=2, pad_h=0),
]


BWD_MODES = {
    # the default path
    "default": {},
    # the split kernels (sample kernel + windowed input kernel), every dtype
    "split": {"bwd_split": 1},
    # the same with a one-pixel halo: most samples leave the window and take
    # the far path
    "split_halo1": {"bwd_split": 1, "bwd_halo": 1},
    # the split kernels with gradient rows written straight to memory and the
    # sample kernel over consecutive items instead of tiles
    "split_direct": {"bwd_split": 1, "bwd_stage": 0, "fwd_tile": 0},
    # the two split kernels as separate launches instead of one
    "split_unfused": {"bwd_split": 1, "bwd_fuse": 0},
    # the single-pass atomic kernels
    "single_pass": {"bwd_split": 0},
    # the split kernels reducing into the float32 accumulator even where one
    # input block covers a whole plane (and would write grad_input directly)
    "split_accumulate": {"bwd_split": 1, "bwd_direct": 0},
}


@pytest.mark.parametrize("w", SPLIT, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", list(BWD_MODES))
def test_backward_paths(w, mode, opts):
    opts.update(BWD_MODES[mode])
    check_bwd(w, make_inputs(w))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["split", "single_pass"])
def test_backward_crowded_samples(dt, mode, opts):
    # every sample of a 32x32 image aimed at one cell: the cells inside each
    # tile's window collect hundreds of samples, the rest leave the window
    opts.update(BWD_MODES[mode])
    w = small(f"crowd_{dt}", dt, gc=16, G=1, N=1, H=32, W=32, softmax=1)
    t = make_inputs(w)
    ho = torch.arange(w.H_out).view(-1, 1, 1)
    wo = torch.arange(w.W_out).view(1, -1, 1)
    taps = torch.tensor(oracle.taps(oracle_params(w)), dtype=torch.float32)   # (P, 2) as (x, y)
    # targets jittered inside the cell [16, 17)^2 so that the samples differ
    # (identical samples would make the DCNv3 mask gradient vanish exactly)
    jit = torch.rand((w.N, w.H_out, w.W_out, w.G, w.P, 2), generator=torch.Generator().manual_seed(3))
    off = torch.empty(w.N, w.H_out, w.W_out, w.G, w.P, 2)
    off[..., 0] = (16.1 - wo - taps[:, 0]).unsqueeze(0).unsqueeze(3) + 0.8 * jit[..., 0]
    off[..., 1] = (16.1 - ho - taps[:, 1]).unsqueeze(0).unsqueeze(3) + 0.8 * jit[..., 1]
    t["offset"] = off.to(t["offset"].dtype)
    check_bwd(w, t)


# ---- hand-worked cases and exact identities -----------------------------------

GOLDEN = json.load(open(os.path.join(HERE, "golden", "hand_cases.json")))


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=[c["name"] for c in GOLDEN["cases"]])
def test_hand_cases_on_gpu(case):
    p = B.Params(dtype=B.DCN_F32, **case["params"])
    f = lambda k: torch.tensor(case[k], dtype=torch.float32, device="cuda")
    out = torch.empty_like(f("output"))
    B.dcn_core_fwd(p, f("input"), f("offset"), f("mask"), out)
    gi, go, gm = (torch.empty_like(f(k)) for k in ("input", "offset", "mask"))
    B.dcn_core_bwd(p, f("grad_out"), f("input"), f("offset"), f("mask"), gi, go, gm)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(out), np.array(case["output"]), rtol=0, atol=1e-6)
    for name, got in (("grad_input", gi), ("grad_offset", go), ("grad_mask", gm)):
        if name in case:
            np.testing.assert_allclose(f64(got), np.array(case[name]), rtol=0, atol=1e-6,
                                       err_msg=name)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("dxy", [(0, 0), (2, -1), (-3, 3)])
def test_integer_offsets_copy_exactly(dt, dxy):
    # one-hot weights and whole-pixel offsets: every output is a copy of an
    # input element (or 0 past the edge), bit for bit, in every dtype
    w = small(f"copy_{dt}", dt, gc=16, G=2, N=2, H=11, W=10, stride_h=2, dilation_w=2, pad_w=2)
    t = make_inputs(w)
    t["offset"] = torch.zeros_like(t["offset"])
    t["offset"][..., 0] = dxy[0]
    t["offset"][..., 1] = dxy[1]
    mask = torch.zeros_like(t["mask"])
    k = 5
    mask[..., k] = 1.0
    t["mask"] = mask
    out = run_fwd(w, t)
    ref = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    np.testing.assert_array_equal(f64(out), ref)


@pytest.mark.parametrize("far", [40.0, -40.0, 1e30, math.inf, -math.inf, math.nan])
def test_out_of_image_samples_are_zero(far):
    w = small("oob", "f32", softmax=1)
    t = make_inputs(w)
    t["offset"][..., 1] = far
    out = run_fwd(w, t)
    assert torch.all(out == 0)
    gi, go, gm = run_bwd(w, t)
    assert torch.all(gi == 0) and torch.all(go == 0) and torch.all(gm == 0)


def test_fp16_huge_offsets_stay_finite():
    # float16 offsets at the top of their range (65504) and infinities
    w = small("f16_huge", "f16")
    t = make_inputs(w)
    t["offset"].view(-1)[::3] = 65504.0
    t["offset"].view(-1)[1::7] = -math.inf
    check_fwd(w, t)
    check_bwd(w, t)


def test_empty_batch():
    w = small("empty", "f16", N=0)
    p = lib_params(w)
    B.dcn_core_fwd(p, None, None, None, None)
    B.dcn_core_bwd(p, None, None, None, None, None, None, None)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_element_aligned_slices_take_the_scalar_path(dt):
    # tensors that start one element past a 16-byte boundary
    w = small(f"misaligned_{dt}", dt, gc=16)
    t = make_inputs(w)
    dev = {}
    for k, v in t.items():
        flat = torch.empty(v.numel() + 2, dtype=v.dtype, device="cuda")
        s = 2 if k == "offset" else 1      # offsets keep their (dx, dy) pairs aligned
        view = flat[s:s + v.numel()].view(v.shape)
        view.copy_(v.cuda())
        dev[k] = view
    p = lib_params(w)
    out = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=t["input"].dtype, device="cuda")
    B.dcn_core_fwd(p, dev["input"], dev["offset"], dev["mask"], out)
    flat = torch.empty(out.numel() + 1, dtype=out.dtype, device="cuda")
    out2 = flat[1:].view(out.shape)
    B.dcn_core_fwd(p, dev["input"], dev["offset"], dev["mask"], out2)
    torch.cuda.synchronize()
    ref = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    assert_close(out, ref, dt, "output")
    assert_close(out2, ref, dt, "misaligned output")


def test_runs_on_the_given_stream():
    w = small("stream", "bf16", softmax=1, N=4)
    t = make_inputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        i, o, m, g = (t[k].cuda() for k in ("input", "offset", "mask", "grad_out"))
        out = B.core_fwd(i, o, m, w.G, **{k: v for k, v in w.params().items()
                                          if k not in ("N", "H", "W", "G", "gc")})
    s.synchronize()
    ref = oracle.forward(oracle_params(w), f64(t["input"]), f64(t["offset"]), f64(t["mask"]))
    assert_close(out, ref, "bf16", "stream output")


def test_autograd_wrapper():
    w = small("autograd", "f32", softmax=1)
    t = make_inputs(w)
    geom = {k: v for k, v in w.params().items() if k not in ("N", "H", "W", "G", "gc")}
    i, o, m = (t[k].cuda().requires_grad_() for k in ("input", "offset", "mask"))
    out = B.dcn_core(i, o, m, w.G, **geom)
    out.backward(t["grad_out"].cuda())
    rgi, rgo, rgm = oracle.backward(oracle_params(w), f64(t["grad_out"]), f64(t["input"]),
                                    f64(t["offset"]), f64(t["mask"]))
    assert_close(i.grad, rgi, "f32", "grad_input")
    assert_close(o.grad, rgo, "f32", "grad_offset")
    assert_close(m.grad, rgm, "f32", "grad_mask")


def test_more_than_2_31_input_elements():
    # 2 x 1024 x 1100 x 1024 fp16 input elements (2.3e9, 4.6 GB); whole-pixel
    # offsets and one-hot weights make each output an exact copy of one input
    # element, checked at sampled pixels, most of them past element 2^31.
    N, H, W, G, gc = 2, 1024, 1100, 4, 256
    C = G * gc
    assert N * H * W * C > 2 ** 31
    p = B.Params(N=N, H=H, W=W, G=G, gc=gc, dtype=B.DCN_F16)
    ho, wo = B.dcn_out_shape(p)
    gen = torch.Generator(device="cuda").manual_seed(5)
    x = (torch.rand((N, H, W, C), generator=gen, device="cuda", dtype=torch.float16) * 2 - 1)
    off = torch.zeros((N, ho, wo, G, 9, 2), dtype=torch.float16, device="cuda")
    off[..., 0] = 1.0
    off[..., 1] = -2.0
    mask = torch.zeros((N, ho, wo, G, 9), dtype=torch.float16, device="cuda")
    mask[..., 8] = 1.0          # tap (+1, +1)
    out = torch.empty((N, ho, wo, C), dtype=torch.float16, device="cuda")
    B.dcn_core_fwd(p, x, off, mask, out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for n, y, xx in zip(rng.integers(0, N, 200), rng.integers(0, ho, 200), rng.integers(0, wo, 200)):
        sy, sx = y + 1 - 2, xx + 1 + 1
        want = x[n, sy, sx] if (0 <= sy < H and 0 <= sx < W) else torch.zeros(C, dtype=x.dtype,
                                                                               device="cuda")
        assert torch.equal(out[n, y, xx], want), (n, y, xx)
    assert torch.equal(out[N - 1, ho - 3, wo - 3], x[N - 1, ho - 4, wo - 1])


def test_no_tensor_copy_wait_ran_out():
    # every tensor copy the tests above waited for arrived in time
    assert B.dcn_wait_timeouts() == 0
