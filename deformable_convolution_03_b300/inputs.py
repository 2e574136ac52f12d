"""Seeded synthetic inputs and the workload table.

This module holds no arithmetic of the deformable aggregation itself: it only
names shapes and draws random tensors.  It is the one module that both the
CUDA-path tests and the oracle tests use, so that both sides see identical
bits.  The output size and the number of sampling points of every workload
are written out as literal numbers (the tests check that the library and the
oracle both derive the same ones).

Workload shapes are those of the FlashInternImage-T stages (channels 64,
groups [4, 8, 16, 32], page "DCNv4高效实践指南：掌握可变形卷积的3倍速度提升技术",
section 图像分类任务配置, at 224x224 input: 56/28/14/7 pixel stages) and of the
InternImage-G first stage (channels 512, groups 16, page
"没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 一).
Value distributions: input U(-1, 1), offsets N(0, s) pixels, mask N(0, 1)
(logits when the op applies a softmax), upstream gradient N(0, 1).  Values are
drawn in float32 and rounded to the storage dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    W: int
    G: int
    gc: int
    H_out: int
    W_out: int
    P: int
    kernel_h: int = 3
    kernel_w: int = 3
    stride_h: int = 1
    stride_w: int = 1
    pad_h: int = 1
    pad_w: int = 1
    dilation_h: int = 1
    dilation_w: int = 1
    offset_scale: float = 1.0
    softmax: int = 0
    remove_center: int = 0
    dtype: str = "f32"
    offset_std: float = 2.0
    backward: bool = False
    seed: int = 1234
    note: str = ""

    @property
    def C(self) -> int:
        return self.G * self.gc

    def params(self) -> dict:
        """Keyword arguments shared by the library's and the oracle's parameter records."""
        return dict(N=self.N, H=self.H, W=self.W, G=self.G, gc=self.gc,
                    kernel_h=self.kernel_h, kernel_w=self.kernel_w,
                    stride_h=self.stride_h, stride_w=self.stride_w,
                    pad_h=self.pad_h, pad_w=self.pad_w,
                    dilation_h=self.dilation_h, dilation_w=self.dilation_w,
                    offset_scale=self.offset_scale, softmax=self.softmax,
                    remove_center=self.remove_center)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _t_stage(i: int, hw: int, c: int, g: int, dtype: str) -> Workload:
    return Workload(name=f"t_stage{i}_{dtype}", N=64, H=hw, W=hw, G=g, gc=c // g,
                    H_out=hw, W_out=hw, P=9, dtype=dtype, softmax=0, offset_std=2.0,
                    seed=1234 + 3, note=f"FlashInternImage-T stage {i}, DCNv4")


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    # DCNv3, tiny, float32
    Workload(name="v3_tiny_f32", N=1, H=8, W=8, G=2, gc=8, H_out=8, W_out=8, P=9,
             softmax=1, dtype="f32", offset_std=2.0, seed=1234 + 1,
             note="DCNv3 tiny, softmax mask"),
    # DCNv4 at FlashInternImage-T stage 1, float16 storage
    Workload(name="t_stage1_f16", N=64, H=56, W=56, G=4, gc=16, H_out=56, W_out=56, P=9,
             softmax=0, dtype="f16", offset_std=2.0, seed=1234 + 2,
             note="FlashInternImage-T stage 1, DCNv4, fp16 storage / fp32 accumulation"),
    # DCNv4 over all four FlashInternImage-T stages, bfloat16
    _t_stage(1, 56, 64, 4, "bf16"),
    _t_stage(2, 28, 128, 8, "bf16"),
    _t_stage(3, 14, 256, 16, "bf16"),
    _t_stage(4, 7, 512, 32, "bf16"),
    # DCNv3 at InternImage-G stage 1, bfloat16; and without the centre tap
    Workload(name="g_stage1_bf16", N=2, H=128, W=128, G=16, gc=32, H_out=128, W_out=128, P=9,
             softmax=1, dtype="bf16", offset_std=2.0, seed=1234 + 4,
             note="InternImage-G stage 1, DCNv3 (softmax)"),
    Workload(name="g_stage1_rc_bf16", N=2, H=128, W=128, G=16, gc=32, H_out=128, W_out=128,
             P=8, softmax=1, remove_center=1, dtype="bf16", offset_std=2.0, seed=1234 + 4,
             note="InternImage-G stage 1, DCNv3, remove_center"),
    # DCNv4 forward + backward, float32, wide offsets
    Workload(name="fb28_f32", N=64, H=28, W=28, G=8, gc=16, H_out=28, W_out=28, P=9,
             softmax=0, dtype="f32", offset_std=3.0, backward=True, seed=1234 + 5,
             note="DCNv4 fwd+bwd, offsets N(0,3): many samples out of bounds"),
    Workload(name="fb28_s2d2_f32", N=64, H=28, W=28, G=8, gc=16, H_out=13, W_out=13, P=9,
             stride_h=2, stride_w=2, pad_h=1, pad_w=1, dilation_h=2, dilation_w=2,
             softmax=0, dtype="f32", offset_std=3.0, backward=True, seed=1234 + 5,
             note="DCNv4 fwd+bwd, stride 2, pad 1, dilation 2"),
]}

# The workloads grouped by what they exercise.
SUITES = {
    "dcnv3_tiny_f32": ["v3_tiny_f32"],
    "dcnv4_t_stage1_f16": ["t_stage1_f16"],
    "dcnv4_t_stages_bf16": ["t_stage1_bf16", "t_stage2_bf16", "t_stage3_bf16", "t_stage4_bf16"],
    "dcnv3_g_stage1_bf16": ["g_stage1_bf16", "g_stage1_rc_bf16"],
    "dcnv4_fwd_bwd_f32": ["fb28_f32", "fb28_s2d2_f32"],
}

# FlashInternImage-T block depths per stage (DEPTHS [4, 4, 18, 4]).
T_DEPTHS = [4, 4, 18, 4]


def make_inputs(w: Workload, seed: int | None = None, grad: bool | None = None) -> dict:
    """Seeded CPU tensors in the storage dtype.

    Returns input (N,H,W,G*gc), offset (N,Ho,Wo,G,P,2), mask (N,Ho,Wo,G,P) and,
    when ``grad`` (default: the workload's backward flag), grad_out
    (N,Ho,Wo,G*gc).  Each tensor has its own sub-seed, so adding a tensor never
    changes the others.
    """
    seed = w.seed if seed is None else seed
    grad = w.backward if grad is None else grad
    dt = DTYPES[w.dtype]

    def gen(k: int) -> torch.Generator:
        return torch.Generator().manual_seed(seed * 16 + k)

    out = {}
    out["input"] = (torch.rand((w.N, w.H, w.W, w.C), generator=gen(0)) * 2 - 1).to(dt)
    out["offset"] = (torch.randn((w.N, w.H_out, w.W_out, w.G, w.P, 2), generator=gen(1))
                     * w.offset_std).to(dt)
    out["mask"] = torch.randn((w.N, w.H_out, w.W_out, w.G, w.P), generator=gen(2)).to(dt)
    if grad:
        out["grad_out"] = torch.randn((w.N, w.H_out, w.W_out, w.C), generator=gen(3)).to(dt)
    return out


def make_dwconv_inputs(N: int, H: int, W: int, C: int, k: int, dtype: str, seed: int = 0,
                       bias: bool = True) -> dict:
    """Seeded CPU tensors for the offset branch's feature step, in the storage
    dtype: x (N,H,W,C) U(-1, 1) like the core's input; the depthwise kernel
    (k,k,C) and bias (C) U(-1/k, 1/k) (a convolution layer's default
    initialisation, fan-in k*k); LayerNorm gamma 1 + N(0, 0.1) and beta
    N(0, 0.1) (its default 1 and 0, perturbed so that both matter)."""
    dt = DTYPES[dtype]

    def gen(j: int) -> torch.Generator:
        return torch.Generator().manual_seed(seed * 16 + 8 + j)

    out = {"x": (torch.rand((N, H, W, C), generator=gen(0)) * 2 - 1).to(dt),
           "weight": ((torch.rand((k, k, C), generator=gen(1)) * 2 - 1) / k).to(dt),
           "gamma": (1 + 0.1 * torch.randn(C, generator=gen(3))).to(dt),
           "beta": (0.1 * torch.randn(C, generator=gen(4))).to(dt)}
    out["bias"] = ((torch.rand(C, generator=gen(2)) * 2 - 1) / k).to(dt) if bias else None
    return out


def ideal_bytes(w: Workload) -> dict:
    """Bytes that must cross HBM at least once: each tensor read or written once.

    forward:  input + offset + mask (read) + output (write)
    backward: grad_out + input + offset + mask (read)
              + grad_input + grad_offset + grad_mask (write)
    """
    es = torch.empty((), dtype=DTYPES[w.dtype]).element_size()
    n_in = w.N * w.H * w.W * w.C
    n_out = w.N * w.H_out * w.W_out * w.C
    n_off = w.N * w.H_out * w.W_out * w.G * w.P * 2
    n_mask = n_off // 2
    fwd = es * (n_in + n_off + n_mask + n_out)
    bwd = es * (n_out + n_in + n_off + n_mask + n_in + n_off + n_mask)
    return {"fwd": fwd, "bwd": bwd}
