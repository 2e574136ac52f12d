/*
 * dcn_oracle.c -- the oracle for the DCNv3 / DCNv4 core deformable aggregation.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct yardstick that
 * the CUDA library is checked against.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load it.  It shares no code, header or
 * constant with the CUDA sources, and nothing in the product path calls it.
 *
 * Arithmetic is binary64 throughout, written as plain nested loops in the order
 * of the steps on the page
 *   "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读"
 *   (the walkthrough of dcnv3_core_pytorch), section 四, steps 1-5:
 *     1. zero-pad the channels-last input by (pad_h, pad_w); the output size
 *        is the one a strided, dilated convolution of that kernel gives;
 *     2. reference point of each output pixel (centre of its receptive field
 *        in the padded input) plus the fixed dilation grid of kernel taps,
 *        the grid scaled by offset_scale;
 *     3. add the predicted offset (pixel units) times offset_scale; with
 *        remove_center the centre tap is dropped, so P = kh*kw - remove_center;
 *     4. bilinear sampling with grid_sample's conventions: align_corners=False
 *        (normalised u maps to pixel u*W_in - 0.5) and padding_mode=zeros;
 *     5. weight each sampled vector by the mask and sum over the P points.
 *   The mask is a softmax over the P points of each (pixel, group) for DCNv3
 *   (same page, section 三 item 3) and the raw mask for DCNv4 (page
 *   "DCNv4高效实践指南：掌握可变形卷积的3倍速度提升技术", section
 *   核心架构与性能优化: the softmax is removed).
 *
 * The backward is the analytic derivative of exactly that forward.
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes of this repository):
 *   - tap order inside the P points: x-major, p = ix*kernel_h + iy (a meshgrid
 *     over the x taps then the y taps), the centre deleted in place when
 *     remove_center is set;
 *   - offset components per point are (dx, dy), grid_sample's (x, y) order;
 *   - pad_h pads the height and pad_w the width;
 *   - a sample whose location (in unpadded pixel units) is not finite or lies
 *     outside the open box (-1, W) x (-1, H) contributes nothing, and has no
 *     gradient (all four of its corners are in the zero padding there);
 *   - at an integer coordinate the cell [x0, x0+1] is used (floor), so the
 *     offset derivative there is the one-sided derivative from the right.
 *
 * Precision of the one integer decision (the cell, floor of the location):
 * with coord_f32 = 0 the location is binary64.  With coord_f32 = 1 the
 * location is first formed in binary32 exactly as the CUDA kernels form it,
 *     b = fmaf(tap, offset_scale, ref)          ref = wo*stride - pad + c
 *     x = fmaf(offset, offset_scale, b)
 * (unpadded pixel units, c = floor(dilation*(k-1)/2)), so that both sides take
 * floor() of the same number; the fraction x - floor(x) is then exact and the
 * rest stays binary64.  Everything else is identical between the two modes.
 */
#include <math.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int N, H, W, G, gc;
  int kernel_h, kernel_w;
  int stride_h, stride_w;
  int pad_h, pad_w;
  int dilation_h, dilation_w;
  double offset_scale;
  int softmax;        /* 1: mask holds logits, softmax over the P points (DCNv3) */
  int remove_center;  /* 1: the centre tap is not sampled */
  int coord_f32;      /* 1: location rounded to binary32 before floor() */
} dcno_params;

#define DCNO_MAX_P 1024

/* ---- step 1: output size and the zero-padded input -------------------- */

/* Output size of a strided, dilated kernel over the padded input.  Returns 0
 * on success, -1 when the parameters are out of range or the output would be
 * empty. */
int dcno_out_shape(const dcno_params* q, int* H_out, int* W_out) {
  if (q->kernel_h < 1 || q->kernel_w < 1 || q->stride_h < 1 || q->stride_w < 1 ||
      q->dilation_h < 1 || q->dilation_w < 1 || q->pad_h < 0 || q->pad_w < 0 ||
      q->H < 1 || q->W < 1)
    return -1;
  if (q->remove_center && ((q->kernel_h % 2) == 0 || (q->kernel_w % 2) == 0)) return -1;
  int Hp = q->H + 2 * q->pad_h, Wp = q->W + 2 * q->pad_w;
  int ext_h = q->dilation_h * (q->kernel_h - 1) + 1;
  int ext_w = q->dilation_w * (q->kernel_w - 1) + 1;
  if (Hp < ext_h || Wp < ext_w) return -1;
  *H_out = (Hp - ext_h) / q->stride_h + 1;
  *W_out = (Wp - ext_w) / q->stride_w + 1;
  return 0;
}

/* The zero-padded input at padded pixel (yp, xp), channel cc of group g:
 * F.pad with zeros, and grid_sample's zero padding beyond the padded frame. */
static double padded_pixel(const dcno_params* q, const double* input, int n, long yp, long xp,
                           int g, int cc) {
  long y = yp - q->pad_h, x = xp - q->pad_w;
  if (y < 0 || y >= q->H || x < 0 || x >= q->W) return 0.0;
  long C = (long)q->G * q->gc;
  return input[(((long)n * q->H + y) * q->W + x) * C + (long)g * q->gc + cc];
}

/* ---- step 2: the dilation grid of taps -------------------------------- */

/* Integer tap positions (in units of pixels, before offset_scale) relative to
 * the reference point, in the x-major order described above.  Returns P. */
int dcno_taps(const dcno_params* q, int* tap_x, int* tap_y) {
  int cw = (q->dilation_w * (q->kernel_w - 1)) / 2;
  int ch = (q->dilation_h * (q->kernel_h - 1)) / 2;
  int P = 0;
  for (int ix = 0; ix < q->kernel_w; ++ix) {
    for (int iy = 0; iy < q->kernel_h; ++iy) {
      if (q->remove_center && ix == (q->kernel_w - 1) / 2 && iy == (q->kernel_h - 1) / 2) continue;
      tap_x[P] = ix * q->dilation_w - cw;
      tap_y[P] = iy * q->dilation_h - ch;
      ++P;
    }
  }
  return P;
}

/* ---- steps 2-3: the sampling location --------------------------------- */

/* Location of point (tap, offset) for output index o along one axis, in
 * padded pixel units as grid_sample(align_corners=False) reads it:
 *   ref   = c + 0.5 + o*stride        (receptive-field centre, padded frame)
 *   u     = (ref + tap*os + off*os) / extent     (normalised, step 3)
 *   pixel = u*extent - 0.5
 * The division by the extent and the multiplication by it cancel, so the
 * pixel is formed directly.  Returned in the unpadded frame (pixel - pad). */
static double location(int o, int stride, int pad, int c, int tap, double off, double os,
                       int coord_f32) {
  if (coord_f32) {
    float ref = (float)(o * stride - pad + c);
    float b = fmaf((float)tap, (float)os, ref);
    return (double)fmaf((float)off, (float)os, b);
  }
  double ref = (double)c + 0.5 + (double)o * stride;
  double pixel = (ref + tap * os + off * os) - 0.5;
  return pixel - pad;
}

/* ---- step 4: bilinear sampling ---------------------------------------- */

typedef struct {
  int valid;           /* 0: the sample contributes nothing */
  long x0, y0;         /* top-left corner, unpadded frame */
  double fx, fy;       /* fractions in [0, 1) */
} dcno_cell;

static dcno_cell cell_of(const dcno_params* q, double x, double y) {
  dcno_cell cl;
  memset(&cl, 0, sizeof cl);
  if (!isfinite(x) || !isfinite(y) || !(x > -1.0) || !(x < q->W) || !(y > -1.0) || !(y < q->H))
    return cl;
  double fx0 = floor(x), fy0 = floor(y);
  cl.valid = 1;
  cl.x0 = (long)fx0;
  cl.y0 = (long)fy0;
  cl.fx = x - fx0;
  cl.fy = y - fy0;
  return cl;
}

/* Value of the zero-padded input at one corner given in the unpadded frame. */
static double corner(const dcno_params* q, const double* input, int n, long y, long x, int g,
                     int cc) {
  return padded_pixel(q, input, n, y + q->pad_h, x + q->pad_w, g, cc);
}

static double bilinear(const dcno_params* q, const double* input, int n, const dcno_cell* cl,
                       int g, int cc) {
  if (!cl->valid) return 0.0;
  double v00 = corner(q, input, n, cl->y0, cl->x0, g, cc);
  double v01 = corner(q, input, n, cl->y0, cl->x0 + 1, g, cc);
  double v10 = corner(q, input, n, cl->y0 + 1, cl->x0, g, cc);
  double v11 = corner(q, input, n, cl->y0 + 1, cl->x0 + 1, g, cc);
  return (1.0 - cl->fy) * ((1.0 - cl->fx) * v00 + cl->fx * v01) +
         cl->fy * ((1.0 - cl->fx) * v10 + cl->fx * v11);
}

/* ---- the modulation weights -------------------------------------------- */

/* m[p] for one (pixel, group): softmax over the P logits (DCNv3) or the raw
 * mask (DCNv4).  The maximum is subtracted before exp(), which leaves the
 * softmax unchanged and keeps exp() finite. */
static void weights(const dcno_params* q, const double* mask_pg, int P, double* m) {
  if (!q->softmax) {
    for (int p = 0; p < P; ++p) m[p] = mask_pg[p];
    return;
  }
  double mx = -INFINITY;
  for (int p = 0; p < P; ++p)
    if (mask_pg[p] > mx) mx = mask_pg[p];
  double s = 0.0;
  for (int p = 0; p < P; ++p) {
    m[p] = exp(mask_pg[p] - mx);
    s += m[p];
  }
  for (int p = 0; p < P; ++p) m[p] /= s;
}

/* ---- step 5: forward ---------------------------------------------------- */

static void forward_pixel(const dcno_params* q, int Ho, int Wo, const int* tx, const int* ty,
                          int P, const double* input, const double* offset, const double* mask,
                          long pix, double* out_pix) {
  int n = (int)(pix / ((long)Ho * Wo));
  int ho = (int)((pix / Wo) % Ho);
  int wo = (int)(pix % Wo);
  int cw = (q->dilation_w * (q->kernel_w - 1)) / 2;
  int ch = (q->dilation_h * (q->kernel_h - 1)) / 2;
  double m[DCNO_MAX_P];
  for (int g = 0; g < q->G; ++g) {
    long unit = pix * q->G + g;
    const double* off = offset + unit * P * 2;
    weights(q, mask + unit * P, P, m);
    for (int cc = 0; cc < q->gc; ++cc) out_pix[(long)g * q->gc + cc] = 0.0;
    for (int p = 0; p < P; ++p) {
      double x = location(wo, q->stride_w, q->pad_w, cw, tx[p], off[2 * p + 0], q->offset_scale,
                          q->coord_f32);
      double y = location(ho, q->stride_h, q->pad_h, ch, ty[p], off[2 * p + 1], q->offset_scale,
                          q->coord_f32);
      dcno_cell cl = cell_of(q, x, y);
      if (!cl.valid) continue; /* contributes nothing, whatever its weight */
      for (int cc = 0; cc < q->gc; ++cc)
        out_pix[(long)g * q->gc + cc] += m[p] * bilinear(q, input, n, &cl, g, cc);
    }
  }
}

/* output[N,Ho,Wo,G*gc] from input[N,H,W,G*gc], offset[N,Ho,Wo,G,P,2],
 * mask[N,Ho,Wo,G,P].  Returns 0, or -1 on invalid parameters. */
int dcno_forward(const dcno_params* q, const double* input, const double* offset,
                 const double* mask, double* output) {
  int Ho, Wo, tx[DCNO_MAX_P], ty[DCNO_MAX_P];
  if (dcno_out_shape(q, &Ho, &Wo) != 0) return -1;
  if ((long)q->kernel_h * q->kernel_w > DCNO_MAX_P) return -1;
  int P = dcno_taps(q, tx, ty);
  long npix = (long)q->N * Ho * Wo;
  long C = (long)q->G * q->gc;
#pragma omp parallel for schedule(static)
  for (long pix = 0; pix < npix; ++pix)
    forward_pixel(q, Ho, Wo, tx, ty, P, input, offset, mask, pix, output + pix * C);
  return 0;
}

/* The forward at a list of flat output pixels (n*Ho*Wo + ho*Wo + wo) only;
 * out receives G*gc values per listed pixel.  For spot checks at sizes where
 * the whole output is not needed. */
int dcno_forward_pixels(const dcno_params* q, const double* input, const double* offset,
                        const double* mask, const long long* pixels, long npix, double* out) {
  int Ho, Wo, tx[DCNO_MAX_P], ty[DCNO_MAX_P];
  if (dcno_out_shape(q, &Ho, &Wo) != 0) return -1;
  if ((long)q->kernel_h * q->kernel_w > DCNO_MAX_P) return -1;
  int P = dcno_taps(q, tx, ty);
  long C = (long)q->G * q->gc;
  long total = (long)q->N * Ho * Wo;
  for (long i = 0; i < npix; ++i)
    if (pixels[i] < 0 || pixels[i] >= total) return -1;
#pragma omp parallel for schedule(static)
  for (long i = 0; i < npix; ++i)
    forward_pixel(q, Ho, Wo, tx, ty, P, input, offset, mask, (long)pixels[i], out + i * C);
  return 0;
}

/* ---- backward ----------------------------------------------------------- */

/* Gradients of L = <grad_out, output> contributed by one output pixel:
 * grad_offset and grad_mask of its G*P points are written to goff_pix and
 * gmask_pix; its scatter into grad_input is added to grad_input (atomically
 * when several threads may add to the same element). */
static void backward_pixel(const dcno_params* q, int Ho, int Wo, const int* tx, const int* ty,
                           int P, const double* grad_out, const double* input,
                           const double* offset, const double* mask, long pix,
                           double* grad_input, double* goff_pix, double* gmask_pix, int atomic) {
  int n = (int)(pix / ((long)Ho * Wo));
  int ho = (int)((pix / Wo) % Ho);
  int wo = (int)(pix % Wo);
  long C = (long)q->G * q->gc;
  int cw = (q->dilation_w * (q->kernel_w - 1)) / 2;
  int ch = (q->dilation_h * (q->kernel_h - 1)) / 2;
  double os = q->offset_scale;
  double m[DCNO_MAX_P], gm[DCNO_MAX_P];
  const double* go = grad_out + pix * C;
  for (int g = 0; g < q->G; ++g) {
    long unit = pix * q->G + g;
    const double* off = offset + unit * P * 2;
    double* goff = goff_pix + (long)g * P * 2;
    weights(q, mask + unit * P, P, m);
    for (int p = 0; p < P; ++p) {
      double x = location(wo, q->stride_w, q->pad_w, cw, tx[p], off[2 * p + 0], os, q->coord_f32);
      double y = location(ho, q->stride_h, q->pad_h, ch, ty[p], off[2 * p + 1], os, q->coord_f32);
      dcno_cell cl = cell_of(q, x, y);
      gm[p] = 0.0;
      goff[2 * p + 0] = 0.0;
      goff[2 * p + 1] = 0.0;
      if (!cl.valid) continue;
      double wx[2] = {1.0 - cl.fx, cl.fx}, wy[2] = {1.0 - cl.fy, cl.fy};
      double dvdx = 0.0, dvdy = 0.0, dv = 0.0;
      for (int cc = 0; cc < q->gc; ++cc) {
        double gcc = go[(long)g * q->gc + cc];
        double v[2][2];
        for (int a = 0; a < 2; ++a)
          for (int b = 0; b < 2; ++b) v[a][b] = corner(q, input, n, cl.y0 + a, cl.x0 + b, g, cc);
        /* d sample / d pixel-x and / d pixel-y, inside the cell */
        double sx = wy[0] * (v[0][1] - v[0][0]) + wy[1] * (v[1][1] - v[1][0]);
        double sy = wx[0] * (v[1][0] - v[0][0]) + wx[1] * (v[1][1] - v[0][1]);
        double s = wy[0] * (wx[0] * v[0][0] + wx[1] * v[0][1]) +
                   wy[1] * (wx[0] * v[1][0] + wx[1] * v[1][1]);
        dv += gcc * s;
        dvdx += gcc * sx;
        dvdy += gcc * sy;
        /* scatter into the input: corners in the zero padding have no input
         * element and receive nothing */
        for (int a = 0; a < 2; ++a)
          for (int b = 0; b < 2; ++b) {
            long yy = cl.y0 + a, xx = cl.x0 + b;
            if (yy < 0 || yy >= q->H || xx < 0 || xx >= q->W) continue;
            double* dst =
                &grad_input[(((long)n * q->H + yy) * q->W + xx) * C + (long)g * q->gc + cc];
            double add = m[p] * wy[a] * wx[b] * gcc;
            if (atomic) {
#pragma omp atomic
              *dst += add;
            } else {
              *dst += add;
            }
          }
      }
      gm[p] = dv;
      /* the location moves by offset_scale per unit of offset */
      goff[2 * p + 0] = os * m[p] * dvdx;
      goff[2 * p + 1] = os * m[p] * dvdy;
    }
    double* gmask = gmask_pix + (long)g * P;
    if (q->softmax) {
      /* d softmax: g_logit_p = m_p * (g_m_p - sum_q m_q g_m_q) */
      double dot = 0.0;
      for (int p = 0; p < P; ++p) dot += m[p] * gm[p];
      for (int p = 0; p < P; ++p) gmask[p] = m[p] * (gm[p] - dot);
    } else {
      for (int p = 0; p < P; ++p) gmask[p] = gm[p];
    }
  }
}

/* Gradients of L = <grad_out, output> with respect to input, offset and mask
 * (the mask logits when softmax is set).  All three outputs are overwritten.
 * Work is split by image n: every scatter into grad_input stays inside the
 * image it came from, so images are independent. */
int dcno_backward(const dcno_params* q, const double* grad_out, const double* input,
                  const double* offset, const double* mask, double* grad_input,
                  double* grad_offset, double* grad_mask) {
  int Ho, Wo, tx[DCNO_MAX_P], ty[DCNO_MAX_P];
  if (dcno_out_shape(q, &Ho, &Wo) != 0) return -1;
  if ((long)q->kernel_h * q->kernel_w > DCNO_MAX_P) return -1;
  int P = dcno_taps(q, tx, ty);
  long C = (long)q->G * q->gc;
  memset(grad_input, 0, sizeof(double) * (size_t)q->N * q->H * q->W * C);
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < q->N; ++n)
    for (long r = 0; r < (long)Ho * Wo; ++r) {
      long pix = (long)n * Ho * Wo + r;
      backward_pixel(q, Ho, Wo, tx, ty, P, grad_out, input, offset, mask, pix, grad_input,
                     grad_offset + pix * q->G * P * 2, grad_mask + pix * q->G * P, 0);
    }
  return 0;
}

/* The backward restricted to the listed output pixels (flat indices as in
 * dcno_forward_pixels): grad_input (full size, overwritten) receives only their
 * scatter; grad_offset and grad_mask receive G*P*2 and G*P values per listed
 * pixel.  For timing on a bounded sample and for spot checks. */
int dcno_backward_pixels(const dcno_params* q, const double* grad_out, const double* input,
                         const double* offset, const double* mask, const long long* pixels,
                         long npix, double* grad_input, double* grad_offset, double* grad_mask) {
  int Ho, Wo, tx[DCNO_MAX_P], ty[DCNO_MAX_P];
  if (dcno_out_shape(q, &Ho, &Wo) != 0) return -1;
  if ((long)q->kernel_h * q->kernel_w > DCNO_MAX_P) return -1;
  int P = dcno_taps(q, tx, ty);
  long C = (long)q->G * q->gc;
  long total = (long)q->N * Ho * Wo;
  for (long i = 0; i < npix; ++i)
    if (pixels[i] < 0 || pixels[i] >= total) return -1;
  memset(grad_input, 0, sizeof(double) * (size_t)q->N * q->H * q->W * C);
#pragma omp parallel for schedule(dynamic, 4)
  for (long i = 0; i < npix; ++i)
    backward_pixel(q, Ho, Wo, tx, ty, P, grad_out, input, offset, mask, (long)pixels[i],
                   grad_input, grad_offset + i * q->G * P * 2, grad_mask + i * q->G * P, 1);
  return 0;
}

/* ---- threads ------------------------------------------------------------- */

void dcno_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int dcno_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
