/*
 * dcn_core.h -- C ABI of the B300 (sm_103a) DCNv3 / DCNv4 core deformable
 * aggregation library (libdcn_b300.so).
 *
 * The operation.  For every output pixel (n, ho, wo), group g and sampling
 * point p the op forms a location from the receptive-field reference point,
 * the dilation grid scaled by offset_scale and the predicted offset scaled by
 * offset_scale; samples the zero-padded channels-last input there bilinearly
 * (grid_sample's align_corners=False, padding_mode=zeros conventions); weights
 * the sampled group vector by the point's modulation weight; and sums over the
 * points.  This is dcnv3_core_pytorch as walked through on the page
 * "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读",
 * section 四 steps 1-5.  The weights are a softmax over the points of each
 * (pixel, group) for DCNv3 (same page, section 三 item 3) and the raw mask
 * for DCNv4 (page "DCNv4高效实践指南：掌握可变形卷积的3倍速度提升技术",
 * section 核心架构与性能优化).
 *
 * In unpadded pixel units, with c_w = floor(dilation_w*(kernel_w-1)/2) and
 * tap t_x = ix*dilation_w - c_w (ix the kernel column):
 *     x = fma(dx, offset_scale, fma(t_x, offset_scale, wo*stride_w - pad_w + c_w))
 * evaluated in binary32, and likewise for y.  Corners outside [0,W)x[0,H)
 * read zero.  A sample whose x is not in (-1, W) or y not in (-1, H) (this
 * includes NaN and infinite offsets) contributes nothing and gets no gradient.
 *
 * Tensors (all channels-last, contiguous, one dtype per call, device memory):
 *     input      (N, H, W, G*gc)
 *     offset     (N, H_out, W_out, G, P, 2)   (dx, dy) in pixels
 *     mask       (N, H_out, W_out, G, P)      logits if softmax, else weights
 *     output     (N, H_out, W_out, G*gc)
 * P = kernel_h*kernel_w - remove_center.  The P points are ordered x-major:
 * p = ix*kernel_h + iy over kernel column ix and row iy, with the centre
 * deleted in place when remove_center is set.
 *
 * Precision.  Storage in float32, float16 or bfloat16; all arithmetic in
 * float32 (fp32 accumulation over points and channels); results rounded to the
 * storage dtype to nearest-even.
 *
 * Ownership and streams.  Every tensor pointer is caller-owned device memory;
 * the library never allocates, frees or retains memory.  Work is enqueued on
 * the caller's cudaStream_t (NULL: the legacy default stream) and the call
 * returns without synchronising: a DCN_OK return covers argument checks and
 * launch errors only.  Calls are safe from several host threads on different
 * streams.  Inputs must not alias outputs.
 *
 * Errors.  Every entry point returns a dcn_status_t (int) and never prints,
 * throws or aborts.  Argument checks run on the host before any CUDA call, so
 * an invalid call has no effect on the device.
 */
#ifndef DCN_CORE_H
#define DCN_CORE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { DCN_F32 = 0, DCN_F16 = 1, DCN_BF16 = 2 } dcn_dtype_t;

typedef enum {
  DCN_OK = 0,
  DCN_ERR_NULL = 1,        /* a required pointer is NULL */
  DCN_ERR_SHAPE = 2,       /* a size or geometry parameter is out of range */
  DCN_ERR_DTYPE = 3,       /* dtype is not a dcn_dtype_t */
  DCN_ERR_ALIGN = 4,       /* a tensor pointer is not aligned to its element size */
  DCN_ERR_UNSUPPORTED = 5, /* valid but not supported by this build (see limits) */
  DCN_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  DCN_ERR_INTERNAL = 7,    /* internal consistency check failed */
  DCN_ERR_WORKSPACE = 8    /* workspace missing or smaller than dcn_core_bwd_workspace() */
} dcn_status_t;

/* Limits of this build. */
#define DCN_MAX_POINTS 64          /* P = kernel_h*kernel_w - remove_center */
#define DCN_MAX_CHANNELS 65536     /* G*gc */

typedef struct {
  int N, H, W;               /* batch and input spatial size, N >= 0, H, W >= 1 */
  int G, gc;                 /* groups and channels per group, >= 1 */
  int kernel_h, kernel_w;    /* >= 1; both odd when remove_center */
  int stride_h, stride_w;    /* >= 1 */
  int pad_h, pad_w;          /* >= 0; pad_h pads the height, pad_w the width */
  int dilation_h, dilation_w;/* >= 1 */
  float offset_scale;        /* scales both the dilation grid and the offsets */
  int softmax;               /* 1: DCNv3, the mask holds logits; 0: DCNv4 raw weights */
  int remove_center;         /* 1: the centre tap is not sampled */
  int dtype;                 /* dcn_dtype_t of every tensor of the call */
} dcn_params_t;

/* Output size: H_out = (H + 2*pad_h - (dilation_h*(kernel_h-1)+1)) / stride_h + 1
 * (integer division), likewise W_out; the size a strided, dilated convolution
 * gives (section 四 step 1 of the walkthrough).  Host only.
 * DCN_ERR_NULL / DCN_ERR_SHAPE / DCN_ERR_DTYPE on bad arguments. */
int dcn_out_shape(const dcn_params_t* p, int* H_out, int* W_out);

/* P, the number of sampling points per (pixel, group), or a negative
 * dcn_status_t on bad arguments.  Host only. */
int dcn_num_points(const dcn_params_t* p);

/* Forward: output = sum_p m_p * bilinear(input, location_p)   (steps 1-5).
 * input, offset, mask: read; output: fully overwritten.  N == 0 launches
 * nothing.  stream: a cudaStream_t. */
int dcn_core_fwd(const dcn_params_t* p, const void* input, const void* offset,
                 const void* mask, void* output, void* stream);

/* Bytes of device workspace dcn_core_bwd needs: N*H*W*G*gc*4 (a float32
 * accumulator for grad_input) for float16 / bfloat16, 0 for float32.
 * Returns 0 as well when the parameters are invalid. */
size_t dcn_core_bwd_workspace(const dcn_params_t* p);

/* Backward of L = <grad_out, output>: the analytic derivative of the forward
 * (the walkthrough's steps 2-5 differentiated; the fused kernel's backward and
 * the memory of its sampling intermediates are discussed on the page
 * "简介这是一份面向图像分类任务实战的FlashInternImage模型资源包", sections 2.2
 * and 5.2, whose kernels recompute the locations instead of storing them).
 *   grad_input  (N, H, W, G*gc)          dL/d input, fully overwritten
 *   grad_offset (N, H_out, W_out, G, P, 2)  dL/d offset, fully overwritten
 *   grad_mask   (N, H_out, W_out, G, P)  dL/d mask; with softmax this is the
 *                                        gradient with respect to the logits
 * At an integer location the cell [x0, x0+1] is used, so the offset gradient
 * there is the one-sided derivative from the right.  grad_input is formed by
 * float32 atomic additions, so its rounding (not its value) depends on the
 * order the GPU runs them in.  workspace: caller-owned device memory of at
 * least dcn_core_bwd_workspace(p) bytes, 16-byte aligned (may be NULL when
 * that is 0); its contents on entry do not matter and on return are
 * unspecified. */
int dcn_core_bwd(const dcn_params_t* p, const void* grad_out, const void* input,
                 const void* offset, const void* mask, void* grad_input, void* grad_offset,
                 void* grad_mask, void* workspace, size_t workspace_bytes, void* stream);

/* DCNv4's merged offset / mask layout: the projection that predicts the
 * offsets and the weights is one linear layer, so they arrive as one tensor
 * (page "告别DCNv3的卡顿：实测DCNv4在A100上3倍提速，手把手教你集成到FlashInternImage",
 * section 1: the offset and weight computations are merged).
 *   offset_mask (N, H_out, W_out, G, row_stride): for each (pixel, group) a
 *   row of 2P offsets ((dx, dy) per point, as in dcn_core_fwd) followed by P
 *   mask values, then row_stride - 3P padding elements (ignored).
 * row_stride >= 3P and even (e.g. 32 for P = 9, a 64-byte row in 16-bit).
 * offset_mask aligned to 2 elements.  Same computation, results and errors as
 * dcn_core_fwd; DCN_ERR_SHAPE for a bad row_stride. */
int dcn_core_fwd_om(const dcn_params_t* p, const void* input, const void* offset_mask,
                    int row_stride, void* output, void* stream);

/* The backward in the merged layout: grad_offset_mask has offset_mask's
 * layout, gradients of the offsets then of the mask (or logits) in each row,
 * and its padding elements are written as zero (the tensor is fully
 * overwritten).  Otherwise as dcn_core_bwd. */
int dcn_core_bwd_om(const dcn_params_t* p, const void* grad_out, const void* input,
                    const void* offset_mask, int row_stride, void* grad_input,
                    void* grad_offset_mask, void* workspace, size_t workspace_bytes,
                    void* stream);

/* Size of the library's own device scratch array used by
 * dcn_core_bwd_noalloc: 32 MiB, enough for the float32 grad_input accumulator
 * of 8M input elements (N*H*W*G*gc <= 8388608). */
#define DCN_NOALLOC_SCRATCH_BYTES (32u << 20)

/* The backward for callers that cannot allocate device memory.  The paper has
 * no counterpart: this entry point exists for deployment, not for the method.
 *
 * Some callers are not allowed to allocate at the point where they run the
 * backward: a plugin inside another runtime that owns all device memory and
 * hands out none during execution, or code with a fixed memory budget that
 * must not grow after start-up (a cudaMalloc there would also synchronise the
 * device).  Such callers cannot provide the workspace dcn_core_bwd needs for
 * float16 / bfloat16.  This entry point computes exactly what dcn_core_bwd
 * computes, with the same arguments minus the workspace, and takes its
 * float32 accumulator from a static array inside the library
 * (DCN_NOALLOC_SCRATCH_BYTES on each GPU where the library's module is
 * loaded, held until the process exits).  The call itself allocates nothing
 * and calls no allocating routine.
 *
 *   - Requests whose dcn_core_bwd_workspace(p) exceeds
 *     DCN_NOALLOC_SCRATCH_BYTES return DCN_ERR_UNSUPPORTED before any CUDA
 *     call; other argument errors are those of dcn_core_bwd.
 *   - The first call on a device (that needs the array: float16 / bfloat16)
 *     looks up the array's device address on the current device, once.  The
 *     array is reserved when the CUDA module holding it is loaded on that
 *     device: with CUDA's default lazy module loading that happens at this
 *     first lookup, so a runtime that hands out all device memory later
 *     should make the first call at start-up (or set
 *     CUDA_MODULE_LOADING=EAGER, which reserves it when the context is
 *     created).  Make that first call before any stream capture.  The stream
 *     must belong to the current device.  cudaDeviceReset invalidates the
 *     remembered address: do not call this entry point on a device after
 *     resetting it.
 *   - All calls on a device share the one array.  Each call clears what it
 *     uses before use, but two calls whose work overlaps on the GPU (different
 *     streams, no ordering between them) race on it and give wrong results:
 *     order them, or use dcn_core_bwd with separate workspaces.
 *   - float32 needs no scratch; the call then behaves as dcn_core_bwd with no
 *     workspace. */
int dcn_core_bwd_noalloc(const dcn_params_t* p, const void* grad_out, const void* input,
                         const void* offset, const void* mask, void* grad_input,
                         void* grad_offset, void* grad_mask, void* stream);

/* The linear projections around the core op: y = x W^T + b, over the rows of
 * a channels-last tensor.  The DCN module feeds the core through such layers:
 * DCNv3's input, offset, mask and output projections (page
 * "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三
 * items 1-6), and DCNv4's one merged offset/mask projection, whose output is
 * the offset_mask tensor of dcn_core_fwd_om when its weight rows are laid out
 * per group as 2P offsets, P mask values and zero padding (page
 * "告别DCNv3的卡顿：实测DCNv4在A100上3倍提速，手把手教你集成到FlashInternImage",
 * section 1).
 *   x     (M, K)  row-major, read
 *   w     (N, K)  row-major (a linear layer's weight), read
 *   bias  (N)     or NULL, read
 *   y     (M, N)  row-major, fully overwritten
 * One dtype for all four.  Arithmetic: float32 accumulation, one rounding to
 * the storage type.  For float16 / bfloat16 with K a multiple of 64, x, w, y
 * 16-byte aligned and N a multiple of 16 from 16 to 256 (K up to 256) or a
 * multiple of 64 (any K), the product runs on the tensor cores (tcgen05,
 * operands staged by tensor copies); otherwise on the CUDA cores
 * (shared-memory tiles).  M == 0 launches nothing.
 * DCN_ERR_NULL / DCN_ERR_SHAPE (M < 0, K < 1, N < 1) / DCN_ERR_DTYPE /
 * DCN_ERR_ALIGN (a pointer not aligned to the element size) on bad
 * arguments, before any CUDA call. */
typedef struct {
  long long M;  /* rows */
  int K, N;     /* input and output features */
  int dtype;    /* dcn_dtype_t of x, w, bias and y */
} dcn_linear_params_t;

int dcn_linear(const dcn_linear_params_t* p, const void* x, const void* w, const void* bias,
               void* y, void* stream);

/* DCNv4's forward with its merged offset/mask projection in the same launch.
 * In the module the offsets and the mask are linear projections of the
 * control features (page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现
 * 逐行解读", section 三 items 3-4), merged by DCNv4 into one layer whose rows
 * are the offset_mask rows of dcn_core_fwd_om (page "告别DCNv3的卡顿：实测DCNv4在
 * A100上3倍提速，手把手教你集成到FlashInternImage", section 1).  This call
 * computes
 *     offset_mask = feat weight^T + bias   (as dcn_linear: float32 sums, one
 *                                           rounding to the storage type)
 *     output      = dcn_core_fwd_om(input, offset_mask, row_stride)
 * where each block of the forward computes its tile's rows on the tensor
 * cores and keeps them in shared memory, so the rows never travel through
 * memory unless asked for.
 *   p            the core's geometry (Ho x Wo output pixels, G groups)
 *   input        (N, H, W, G*gc) channels-last, read
 *   feat         (N, Ho, Wo, K) the projection's input, read
 *   weight       (G*row_stride, K) row-major, read; bias (G*row_stride) or NULL
 *   row_stride   >= 3P and even, as dcn_core_fwd_om (rows: 2P offsets, P mask
 *                values, padding)
 *   output       (N, Ho, Wo, G*gc), fully overwritten
 *   offset_mask  (N, Ho, Wo, G, row_stride) or NULL: when given, the rows are
 *                also written there (the backward needs them)
 * One dtype for all.  With offset_mask given, the call runs dcn_linear into
 * offset_mask and then dcn_core_fwd_om: two launches, measured faster than
 * the single one at every shape tried.  Without it, the single launch runs;
 * it applies to float16 / bfloat16 with K a multiple of 64 up to 256,
 * row_stride a multiple of 8, feat and weight 16-byte aligned and the input
 * laid out for the tensor-copy forward, and other calls without offset_mask
 * return DCN_ERR_UNSUPPORTED.  Both ways compute the same rows (bit for bit)
 * and the same forward on them.
 * Errors as dcn_core_fwd_om, plus DCN_ERR_SHAPE for K < 1. */
int dcn_core_fwd_proj(const dcn_params_t* p, const void* input, const void* feat, int K,
                      const void* weight, const void* bias, int row_stride, void* output,
                      void* offset_mask, void* stream);

/* The centre feature scale between the core op and output_proj (page
 * "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三
 * item 5; page "DCNv4高效实践指南：掌握可变形卷积的3倍速度提升技术", section
 * "高级配置参数详解"): a sigmoid gate mixes the core's output with the centre
 * pixel's projected feature x_proj (the core's input at the same pixel).  One
 * gate per (pixel, group), s = 1 / (1 + exp(-logit)), over the group's
 * gc = C / G channels:
 *     out = core * (1 - s) + x_proj * s
 * and the backward
 *     grad_core = g * (1 - s),  grad_x_proj = g * s,
 *     grad_logits = s (1 - s) * sum over the group's channels of g * (x_proj - core).
 *   core, x_proj, out, grad_out, grad_core, grad_x_proj   (M, C) row-major
 *   logits, grad_logits                                    (M, G) row-major
 * M rows (pixels, N * Ho * Wo), C = G * gc channels, one dtype for all.
 * Arithmetic in float32, one rounding to the storage type (the logit gradient
 * sums its gc products in float32).  out may be the same buffer as core or as
 * x_proj, and grad_core the same as grad_out (in place); other overlaps are
 * not allowed.  Outputs are fully overwritten; M == 0 launches nothing.
 * DCN_ERR_NULL / DCN_ERR_SHAPE (M < 0, C < 1, G < 1, C % G != 0) /
 * DCN_ERR_DTYPE / DCN_ERR_ALIGN (a pointer not aligned to the element size)
 * / DCN_ERR_UNSUPPORTED (M * C >= 2^40) before any CUDA call. */
typedef struct {
  long long M;  /* rows */
  int C, G;     /* channels per row, groups */
  int dtype;    /* dcn_dtype_t of every tensor */
} dcn_cfs_params_t;

int dcn_center_feature_scale(const dcn_cfs_params_t* p, const void* core, const void* x_proj,
                             const void* logits, void* out, void* stream);
int dcn_center_feature_scale_bwd(const dcn_cfs_params_t* p, const void* grad_out,
                                 const void* core, const void* x_proj, const void* logits,
                                 void* grad_core, void* grad_x_proj, void* grad_logits,
                                 void* stream);

/* The core op followed by the centre feature scale in one call, x_proj being
 * the core's own input (the two sections cited above dcn_core_fwd and
 * dcn_center_feature_scale): per (pixel, group) unit,
 *     out = core * (1 - s) + input[n, ho, wo, g, :] * s,  s = 1 / (1 + exp(-logit)),
 * which needs an output the input's size: stride 1 and padding
 * dilation * (kernel - 1) / 2 on both axes (H_out == H, W_out == W).
 *   input, offset, mask   as dcn_core_fwd
 *   logits                (N, H_out, W_out, G), one per unit, read
 *   output                (N, H_out, W_out, G*gc), fully overwritten; must not
 *                         overlap the other tensors
 * For float16 / bfloat16 with separate offset / mask tensors and the input
 * laid out for the tensor-copy forward, one launch: the gate is applied to the
 * core's float32 sums before their one rounding, with x_proj read from the
 * block's staged input window.  Otherwise (float32, other layouts) two
 * launches, dcn_core_fwd into output and dcn_center_feature_scale over it in
 * place, whose core is rounded to the storage type first; the two ways agree
 * within that one extra rounding.
 * The pre-gate core output is never materialised, so this is the inference
 * form: the gate's backward (dcn_center_feature_scale_bwd) needs that core
 * output, which a training step gets from dcn_core_fwd followed by
 * dcn_center_feature_scale.
 * Errors as dcn_core_fwd, plus DCN_ERR_SHAPE when the output is not the
 * input's size, DCN_ERR_NULL / DCN_ERR_ALIGN for logits. */
int dcn_core_fwd_cfs(const dcn_params_t* p, const void* input, const void* offset,
                     const void* mask, const void* logits, void* output, void* stream);

/* The core op followed by the module's output projection in one call (page
 * "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三
 * item 6: output_proj, a linear layer over the core's channels), optionally
 * with the centre feature scale between them (logits non-NULL, as
 * dcn_core_fwd_cfs):
 *     y[n, ho, wo, :] = out[n, ho, wo, :] W^T + bias
 * with out the core's (or the gate's) output rounded to the storage type, as
 * dcn_core_fwd / dcn_core_fwd_cfs store it.
 *   input, offset, mask   as dcn_core_fwd
 *   logits                (N, H_out, W_out, G), or NULL for no gate
 *   weight                (n_out, C) row-major; bias (n_out) or NULL
 *   y                     (N, H_out, W_out, n_out), fully overwritten
 *   scratch               (N, H_out, W_out, C) or NULL: room for out
 * With scratch, out is written there and projected by the kernels of
 * dcn_linear, which read it back from L2 (the faster way).  Without scratch,
 * for float16 / bfloat16 with C = 64 (every channel of a pixel in one block of
 * the tensor-copy forward), separate offset / mask tensors, n_out a multiple
 * of 16 up to 128 and weight and y 16-byte aligned, one launch needs no room
 * for out: the forward's epilogue runs the projection on the tensor cores
 * (tcgen05); any other call without scratch returns DCN_ERR_UNSUPPORTED.
 * Both ways take the same products of the same rounded values with float32
 * sums.  No tensor may overlap another.
 * Errors as dcn_core_fwd (and dcn_core_fwd_cfs with logits), plus
 * DCN_ERR_SHAPE for n_out < 1 and DCN_ERR_NULL for weight or y. */
int dcn_core_fwd_out(const dcn_params_t* p, const void* input, const void* offset,
                     const void* mask, const void* logits, const void* weight, const void* bias,
                     int n_out, void* y, void* scratch, void* stream);

/* The feature step of the DCN module's offset branch (page
 * "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 三
 * item 2: the control features x1 from which the offset and mask projections
 * are computed come from a depthwise convolution, LayerNorm and GELU of the
 * module's input; the page's configuration table gives dw_kernel_size 5).
 * One pass computes, per image n, pixel (i, j) and channel c,
 *     u[c] = bias[c] + sum_{a,e < k} weight[a, e, c] * x[n, i+a-r, j+e-r, c]
 *            (r = (k - 1) / 2, x zero outside the image: the output keeps the
 *            input's size),
 *     z[c] = (u[c] - mean(u)) / sqrt(var(u) + eps) * gamma[c] + beta[c]
 *            (mean and biased variance over the pixel's C channels),
 *     y[n, i, j, c] = z / 2 * (1 + erf(z / sqrt(2)))   (the exact GELU).
 *   x       (N, H, W, C) channels-last, read
 *   weight  (k, k, C)    the depthwise kernel, weight[a, e, c] = a PyTorch
 *                        Conv2d(groups=C) weight[c, 0, a, e], read
 *   bias    (C) or NULL (no bias), read
 *   gamma, beta (C)      the LayerNorm affine parameters, read
 *   y       (N, H, W, C) fully overwritten; must not overlap x
 * One dtype for all.  Arithmetic in float32 (the convolution's k*k products
 * summed in float32, the statistics over float32 sums), one rounding to the
 * storage type; erf is evaluated by Abramowitz and Stegun's formula 7.1.26
 * (absolute error at most 1.5e-7), so GELU is within |z| * 1e-7 of exact
 * before rounding.  The library picks a tiled kernel for k of 3 or 5 with C
 * of 64, 128, 256 or 512, x 16-byte aligned and the other tensors aligned
 * to two elements; any other shape within the limits takes a slower kernel
 * with the same arithmetic.  N == 0 launches nothing.
 * DCN_ERR_NULL / DCN_ERR_DTYPE / DCN_ERR_SHAPE (N < 0, H < 1, W < 1, C < 1,
 * k even, k < 1 or k > DCN_DW_MAX_KERNEL, eps negative or not finite) /
 * DCN_ERR_ALIGN (a pointer not aligned to the element size) /
 * DCN_ERR_UNSUPPORTED (C > DCN_DW_MAX_CHANNELS, N * H * W * C >= 2^40) before
 * any CUDA call. */
#define DCN_DW_MAX_KERNEL 31
#define DCN_DW_MAX_CHANNELS 2048

typedef struct {
  int N, H, W, C;  /* images, height, width, channels */
  int k;           /* kernel size (odd) */
  float eps;       /* LayerNorm epsilon */
  int dtype;       /* dcn_dtype_t of every tensor */
} dcn_dwconv_params_t;

int dcn_dwconv_ln_gelu(const dcn_dwconv_params_t* p, const void* x, const void* weight,
                       const void* bias, const void* gamma, const void* beta, void* y,
                       void* stream);

/* Diagnostics of the asynchronous tensor copies and tensor-core operations
 * some kernels use: the number of thread blocks, since the library was
 * loaded, whose bounded wait for such a copy or operation ran out on the
 * current device.  A block of the tensor-copy forward then computed its
 * results from global memory, so they stay correct; a block of a projection
 * (dcn_linear, dcn_core_fwd_proj) computed nothing, so its outputs are not
 * valid.  A non-zero count means a copy took seconds, i.e. something is wrong
 * with the device.  Reads device counters synchronously (the current device).
 * DCN_ERR_NULL for a NULL count, DCN_ERR_CUDA if the read fails. */
int dcn_wait_timeouts(unsigned long long* count);

/* A static, human-readable name for a dcn_status_t. */
const char* dcn_status_str(int status);

/* Library version, major*10000 + minor*100 + patch. */
int dcn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DCN_CORE_H */
