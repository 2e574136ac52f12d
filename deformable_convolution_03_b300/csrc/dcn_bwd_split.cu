// dcn_bwd_split.cu -- the backward as two kernels with disjoint jobs.
//
// The backward of the core op has two halves that need different hardware:
//
//   * the sample half (grad_offset, grad_mask) gathers the four bilinear
//     corners of every sample, exactly like the forward, and reduces them
//     against grad_out: d_k = sum_c gout_c * corner_k,c.  It wants all of L1
//     for the corner lines and many warps in flight;
//   * the input half (grad_input) is the transpose of the forward's gather:
//     input pixel q receives m * w_k(q) * gout[u] from every sample (u, p)
//     whose bilinear cell has q as corner k.  It never reads the input
//     tensor, but scattering it sample by sample means one float32 reduction
//     into L2 per (sample, corner, channel), and L2 reductions are the
//     slowest resource on this GPU.
//
// bwd_sample_kernel does the first half with the forward's thread layout and
// no grad_input work.  bwd_input_kernel does the second: a CTA owns TH x TW
// output pixels of one (image, group), bins their samples by bilinear cell in
// shared memory (integer counting sort), and sums each pixel of a window
// around the tile's footprint in registers before one vector reduction per
// four channels, about ten times fewer reductions than scattering.  It reads
// only offsets, masks and grad_out.
//
// Derivatives (the analytic derivative of dcnv3_core_pytorch, page
// "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 四
// steps 2-5), with (gx, gy) = (1 - fx, 1 - fy):
//   dL/dm         = gy*(gx*d00 + fx*d01) + fy*(gx*d10 + fx*d11)
//   dL/d offset_x = scale * m * (gy*(d01 - d00) + fy*(d11 - d10))
//   dL/d offset_y = scale * m * (gx*(d10 - d00) + fx*(d11 - d01))
//   (DCNv3)  dL/d logit_p = m_p * (dL/dm_p - sum_q m_q dL/dm_q)
// Corners outside the image read zero, so their d_k is zero and they receive
// nothing.
#include <cuda.h>

#include <climits>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"
#include "dcn_options.h"

namespace dcn {

// ---- the sample half --------------------------------------------------------
// One thread per (unit, slice of CPT channels), slices of 16 to 64 bytes, in
// the wide forward's order: 2-D tiles of output pixels with all groups and
// slices of each (kp.tile_w > 0), else consecutive items.  The unit's
// gc/CPT threads are adjacent lanes; they sum d_k by shuffles and the first
// of them writes the unit's gradients.  With la > 0 those rows are put
// together in shared memory (la elements per unit for the offset rows, lb for
// the mask rows; for the merged layout la is the row stride and lb is 0) and
// written out row by row of the tile with 16-byte stores.
template <typename T, int CPT, int KP>
__device__ __forceinline__ void sample_block(const KParams& kp, const T* __restrict__ gout,
                                             const T* __restrict__ input,
                                             const T* __restrict__ offset,
                                             const T* __restrict__ mask, T* __restrict__ goff,
                                             T* __restrict__ gmask, int la, int lb,
                                             const unsigned bid) {
  constexpr int NW = CPT * (int)sizeof(T) / 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int chunks = kp.gc / CPT;
  const int P = KP > 0 ? KP : kp.P;
  uint32_t unit = 0, n;
  int c0, g, ho, wo, ho0 = 0, wo0 = 0;
  bool active;
  if (kp.tile_w > 0) {
    // tid = (pixel-in-tile * G + g) * chunks + slice
    const int per_px = kp.G * chunks;
    const int lp = threadIdx.x / per_px, r = threadIdx.x - lp * per_px;
    g = r / chunks;
    c0 = (r - g * chunks) * CPT;
    const int tiles = kp.tiles_w * kp.tiles_h;
    n = bid / tiles;
    const int t = bid - n * tiles;
    const int ty = t / kp.tiles_w;
    ho0 = ty * kp.tile_h;
    wo0 = (t - ty * kp.tiles_w) * kp.tile_w;
    ho = ho0 + lp / kp.tile_w;
    wo = wo0 + lp % kp.tile_w;
    active = lp < kp.tile_w * kp.tile_h && ho < kp.Ho && wo < kp.Wo;
    if (active) unit = ((n * (uint32_t)kp.Ho + ho) * kp.Wo + wo) * kp.G + g;
  } else {
    const uint32_t item = bid * blockDim.x + threadIdx.x;
    active = item < (uint32_t)(kp.units * chunks);
    const uint32_t it = active ? item : 0;
    unit = chunks == 1 ? it : it / (uint32_t)chunks;
    c0 = (int)(it - unit * chunks) * CPT;
    const uint32_t q1 = kp.div_G.div(unit);
    g = (int)(unit - q1 * (uint32_t)kp.G);
    const uint32_t q2 = kp.div_Wo.div(q1);
    wo = (int)(q1 - q2 * (uint32_t)kp.Wo);
    n = kp.div_Ho.div(q2);
    ho = (int)(q2 - n * (uint32_t)kp.Ho);
  }
  const bool leader = active && c0 == 0;

  const T* mrow = mask + (size_t)unit * kp.os_mask;
  const T* orow = offset + (size_t)unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow)) {  // (checked build) read unit 0's rows
    mrow = mask;
    orow = offset;
  }
  const T* img = input + (size_t)n * kp.H * kp.W * kp.C + g * kp.gc + c0;
  const uint32_t W = kp.W, H = kp.H, C = kp.C, WC = (uint32_t)kp.W * kp.C;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  uint32_t gw[NW];
  if (active && out_in(kp, gout, gout + (size_t)unit * kp.gc + c0, CPT)) {
    ldg_words<NW>(gout + (size_t)unit * kp.gc + c0, gw);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) gw[i] = 0u;
  }
  Halves<NW> gh;
  if constexpr (sizeof(T) == 2) gh.split(gw);

  // separate offset / mask tensors and a compile-time point count: the rows
  // with a few aligned vector loads
  UnitRows<T, KP> rows;
  bool vec = false;
  // (not for 64-byte float32 slices, whose corners already fill the registers)
  constexpr bool kVecRows = KP > 0 && (sizeof(T) == 2 || CPT <= 8);
  if constexpr (kVecRows) {
    if (!kp.merged) {
      vec = active && rows.load(offset, mask, kp.units, orow, mrow);
    } else if constexpr (KP == 9 && sizeof(T) == 2) {
      // DCNv4's merged 64-byte rows: the whole row in two 256-bit loads
      if (active && kp.merged_rows64 &&
          DCN_IN_SPAN(orow, 64, offset, offset_bytes<T>(kp), kBadRow)) {
        rows.load_merged64(orow);
        vec = true;
      }
    }
  }

  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) {
    mx = -INFINITY;
    if (vec) {
#pragma unroll
      for (int p = 0; p < (KP > 0 ? KP : 1); ++p) mx = fmaxf(mx, rows.msk(p));
      float s = 0.f;
#pragma unroll
      for (int p = 0; p < (KP > 0 ? KP : 1); ++p) s += expf(rows.msk(p) - mx);
      inv = 1.f / s;
    } else {
      for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(mrow + p));
      float s = 0.f;
      for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(mrow + p) - mx);
      inv = 1.f / s;
    }
  }

  // the unit's gradient rows: staged in shared memory, or straight to memory
  const int lu = threadIdx.x / chunks;
  const int ub = blockDim.x / chunks;
  T* s_rows = reinterpret_cast<T*>(smem);
  const int ls = stage_stride(la, (int)sizeof(T));  // the offset rows' staging stride
  T* ro = la > 0 ? s_rows + lu * ls : goff + (size_t)unit * kp.os_off;
  T* rm = la > 0 ? (kp.merged ? ro + 2 * P : s_rows + ub * ls + lu * lb)
                 : gmask + (size_t)unit * kp.os_mask;

  float gm_row[KP > 0 ? KP : DCN_MAX_POINTS];
  float dot = 0.f;

#pragma unroll(KP > 0 ? KP : 1)
  for (int p = 0; p < P; ++p) {
    float m = 0.f;
    float2 d = make_float2(0.f, 0.f);
    if (KP > 0 && vec) {
      m = rows.msk(KP > 0 ? p : 0);
      d = rows.off(KP > 0 ? p : 0);
    } else if (active) {
      m = ld_once_1(mrow + p);
      d = ld_once_2(orow + 2 * p);
    }
    if (kp.softmax) m = expf(m - mx) * inv;
    float x = location(d.x, kp.tap_x[p], scale, ref_x);
    float y = location(d.y, kp.tap_y[p], scale, ref_y);
    const bool valid = active && in_box(x, y, kp.W, kp.H);
    if (!valid) {  // also NaN / inf: the sample contributes nothing
      x = -4.f;
      y = -4.f;
    }
    const float xf = floorf(x), yf = floorf(y);
    const int x0 = (int)xf, y0 = (int)yf;
    const float fx = x - xf, fy = y - yf;
    const bool vx0 = (uint32_t)x0 < W, vx1 = (uint32_t)(x0 + 1) < W;
    const bool vy0 = (uint32_t)y0 < H, vy1 = (uint32_t)(y0 + 1) < H;
    // clamped corners: always inside the image; a corner really outside it
    // reads zero, i.e. its dot product is dropped
    const uint32_t xa = min((uint32_t)x0, W - 1), xb = min((uint32_t)(x0 + 1), W - 1);
    const uint32_t ya = min((uint32_t)y0, H - 1), yb = min((uint32_t)(y0 + 1), H - 1);
    const uint32_t off[4] = {ya * WC + xa * C, ya * WC + xb * C, yb * WC + xa * C,
                             yb * WC + xb * C};
    const bool ok[4] = {vy0 && vx0, vy0 && vx1, vy1 && vx0, vy1 && vx1};
    uint32_t v[4][NW];
#pragma unroll
    for (int k = 0; k < 4; ++k) ldg_words_in<NW>(img + off[k], v[k], input, input_bytes<T>(kp));
    float dk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float s[2] = {0.f, 0.f};
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < NW; ++i) dot_split<T>(s[0], s[1], v[k][i], gh.lo[i], gh.hi[i]);
      } else {
#pragma unroll
        for (int i = 0; i < NW; ++i)
          s[i & 1] = fmaf(__uint_as_float(gw[i]), __uint_as_float(v[k][i]), s[i & 1]);
      }
      dk[k] = ok[k] ? s[0] + s[1] : 0.f;
    }
    for (int s = 1; s < chunks; s <<= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) dk[k] += __shfl_xor_sync(0xffffffffu, dk[k], s);
    }
    if (leader) {
      float gm = 0.f, gox = 0.f, goy = 0.f;
      if (valid) {
        const float gx = 1.f - fx, gy = 1.f - fy;
        gm = gy * (gx * dk[0] + fx * dk[1]) + fy * (gx * dk[2] + fx * dk[3]);
        gox = scale * m * (gy * (dk[1] - dk[0]) + fy * (dk[3] - dk[2]));
        goy = scale * m * (gx * (dk[2] - dk[0]) + fx * (dk[3] - dk[1]));
      }
      ro[2 * p] = Dt<T>::from_f(gox);
      ro[2 * p + 1] = Dt<T>::from_f(goy);
      if (kp.softmax) {
        gm_row[p] = gm;
        dot = fmaf(m, gm, dot);
      } else {
        rm[p] = Dt<T>::from_f(gm);
      }
    }
  }
  if (leader && kp.softmax) {
#pragma unroll(KP > 0 ? KP : 1)
    for (int p = 0; p < P; ++p) {
      const float l = KP > 0 && vec ? rows.msk(KP > 0 ? p : 0) : Dt<T>::one(mrow + p);
      const float m = expf(l - mx) * inv;
      rm[p] = Dt<T>::from_f(m * (gm_row[p] - dot));
    }
  }
  if (leader && kp.merged)
    for (int i = 3 * P; i < kp.os_off; ++i) ro[i] = Dt<T>::from_f(0.f);
  if (la <= 0) return;

  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  constexpr int es = (int)sizeof(T);
  if (kp.tile_w > 0) {
    // tile row ty holds units (n, ho0 + ty, wo0 .. wo0 + nw - 1, all groups),
    // contiguous in memory and in shared memory
    const int nw = min(kp.tile_w, kp.Wo - wo0);
    for (int ty = warp; ty < kp.tile_h; ty += nwarp) {
      const int hh = ho0 + ty;
      if (hh >= kp.Ho) break;
      const size_t u0 = (((size_t)n * kp.Ho + hh) * kp.Wo + wo0) * kp.G;
      const int cnt = nw * kp.G, l0 = ty * kp.tile_w * kp.G;
      if (ls == la)
        warp_copy_out(goff + u0 * kp.os_off, s_rows + l0 * la, cnt * la * es, lane);
      else
        warp_copy_rows_out(goff + u0 * kp.os_off, s_rows + l0 * ls, cnt, la * es, ls * es, lane);
      if (lb > 0)
        warp_copy_out(gmask + u0 * kp.os_mask, s_rows + ub * ls + l0 * lb, cnt * lb * es, lane);
    }
  } else {
    const long long u0 = (long long)bid * ub;
    const int cnt = (int)min((long long)ub, kp.units - u0);
    if (cnt > 0 && warp == 0) {
      if (ls == la)
        warp_copy_out(goff + u0 * kp.os_off, s_rows, cnt * la * es, lane);
      else
        warp_copy_rows_out(goff + u0 * kp.os_off, s_rows, cnt, la * es, ls * es, lane);
    } else if (cnt > 0 && warp == 1 && lb > 0) {
      warp_copy_out(gmask + u0 * kp.os_mask, s_rows + ub * ls, cnt * lb * es, lane);
    }
  }
}

template <typename T, int CPT, int KP>
__global__ void __launch_bounds__(256, sizeof(T) == 2 ? 3 : 2)
bwd_sample_kernel(const KParams kp, const T* __restrict__ gout, const T* __restrict__ input,
                  const T* __restrict__ offset, const T* __restrict__ mask,
                  T* __restrict__ goff, T* __restrict__ gmask, int la, int lb) {
  sample_block<T, CPT, KP>(kp, gout, input, offset, mask, goff, gmask, la, lb, blockIdx.x);
}


// ---- the input half ---------------------------------------------------------
// A CTA owns TH x TW <= blockDim.x output pixels of one (image, group); a
// unit's gc channels are NW words (16, 32 or 64 bytes) and its P <= 16 points.
//   1. one thread per unit: the locations and each sample's bilinear cell
//      relative to the window.  A sample inside the window takes a rank in
//      its cell from a shared-memory integer atomic; a sample whose cell
//      leaves the window ("far", rare) is reduced into memory directly.  The
//      unit's grad_out goes to shared memory.
//      Each in-window sample's four corner weights m*w_k go to shared memory
//      in sample order (unit-major).
//   2. an exclusive scan of the cell counts gives each cell's list head; each
//      sample's id goes to slot head + rank (a counting sort by cell).
//   3. one thread per window pixel: the pixel is a corner of four cells, two
//      adjacent cells in the row above it and two in its own row, so its
//      contributions are two contiguous ranges of the sorted lists, walked in
//      one loop; the sum of w * grad_out over them stays in float32
//      registers, then one vector reduction per four channels goes to
//      memory, only for pixels that received something.
// Windows of neighbouring CTAs overlap, so the accumulator is cleared before
// the launch and reduced into; the kernel never reads it, so its reductions
// carry no memory clobber.  In 16-bit storage each weight is rounded to
// the storage type once and multiplied exactly into the float32 sum
// (mixed-precision FMA), as in the forward.
template <typename T, int NW, int KP>
__device__ __forceinline__ void input_block(const KParams& kp, const WinGeom& wg,
                                            const T* __restrict__ gout,
                                            const T* __restrict__ offset,
                                            const T* __restrict__ mask, float* __restrict__ gin,
                                            T* __restrict__ gdirect, const unsigned bid) {
  constexpr int CPT = NW * 4 / (int)sizeof(T);  // = gc
  constexpr int KPN = KP > 0 ? KP : 16;
  constexpr bool k16 = sizeof(T) == 2;
  // the four weights of a sample: 4 x 16 bits, or 4 x float32; and the two of
  // one row of its corners: (x0, x1) as 2 x 16 bits or 2 x float32
  using Wq = typename std::conditional<k16, uint2, float4>::type;
  using Wh = typename std::conditional<k16, uint32_t, float2>::type;
  extern __shared__ __align__(128) unsigned char smem[];
  const int P = KP > 0 ? KP : kp.P;
  const int nunit = wg.TH * wg.TW;
  const int nsamp = nunit * P;
  const int cw = wg.WW - 1, ncell = (wg.WH - 1) * cw;
  auto up16 = [](int b) { return (b + 15) & ~15; };
  // in cell order: the weights of the corner row y0 + 1 (wa) and y0 (wb), and
  // the sample's unit in the tile
  Wh* wa = reinterpret_cast<Wh*>(smem);                                  // nsamp
  Wh* wb = wa + nsamp;                                                   // nsamp
  unsigned short* eu = reinterpret_cast<unsigned short*>(
      smem + up16(nsamp * (int)sizeof(Wq)));                             // nsamp
  uint32_t* gos = reinterpret_cast<uint32_t*>(
      reinterpret_cast<unsigned char*>(eu) + up16(nsamp * 2));           // nunit * NW
  int* count = reinterpret_cast<int*>(gos + nunit * NW);                 // ncell
  int* head = count + ncell;                                             // ncell + 1
  int* wsum = head + ncell + 1;                                          // 32

  // block = (image, tile, group) with the group fastest, so that the CTAs of
  // one tile read neighbouring sectors of the same lines at about one time
  const int g = bid % kp.G;
  const int rest = bid / kp.G;
  const int tiles = wg.tiles_h * wg.tiles_w;
  const int t = rest % tiles, n = rest / tiles;
  const int th = t / wg.tiles_w, tw = t - th * wg.tiles_w;
  const int ho0 = th * wg.TH, wo0 = tw * wg.TW;
  const int wy0 = ho0 * kp.stride_h + wg.org_y, wx0 = wo0 * kp.stride_w + wg.org_x;

  // ---- pass 1 -------------------------------------------------------------
  const int local = threadIdx.x;
  const int lh = local / wg.TW, lw = local - lh * wg.TW;
  const int ho = ho0 + lh, wo = wo0 + lw;
  const bool active = local < nunit && ho < kp.Ho && wo < kp.Wo;
  const size_t unit = active ? (((size_t)n * kp.Ho + ho) * kp.Wo + wo) * kp.G + g : 0;
  const T* mrow = mask + unit * kp.os_mask;
  const T* orow = offset + unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow)) {  // (checked build) read unit 0's rows
    mrow = mask;
    orow = offset;
  }
  const size_t img_off = (size_t)n * kp.H * kp.W * kp.C + (size_t)g * kp.gc;
  const size_t gin_bytes = input_bytes<float>(kp);
  const int W = kp.W, H = kp.H;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  uint32_t gw[NW];
  if (active && out_in(kp, gout, gout + unit * kp.gc, CPT)) {
    ldg_words<NW>(gout + unit * kp.gc, gw);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) gw[i] = 0u;
  }
  // the unit's offsets and weights, all loads issued before any use and before
  // the barrier that follows the count clear, whose wait then overlaps their
  // latency (stage 1 backward 267 -> 265 us)
  float2 dd[KPN];
  float mm[KPN];
  {
    bool done = false;
    if constexpr (KP > 0) {
      UnitRows<T, KP> rows;
      bool got = false;
      if (active && !kp.merged) {
        got = rows.load(offset, mask, kp.units, orow, mrow);
      } else if constexpr (KP == 9 && sizeof(T) == 2) {
        if (active && kp.merged_rows64 &&
            DCN_IN_SPAN(orow, 64, offset, offset_bytes<T>(kp), kBadRow)) {
          rows.load_merged64(orow);
          got = true;
        }
      }
      if (got) {
#pragma unroll
        for (int p = 0; p < KP; ++p) {
          dd[p] = rows.off(p);
          mm[p] = rows.msk(p);
        }
        done = true;
      }
    }
    if (!done) {
#pragma unroll(KP > 0 ? KP : 1)
      for (int p = 0; p < P; ++p) {
        dd[p] = active ? ld_once_2(orow + 2 * p) : make_float2(0.f, 0.f);
        mm[p] = active ? ld_once_1(mrow + p) : 0.f;
      }
    }
  }
  for (int i = threadIdx.x; i < ncell; i += blockDim.x) count[i] = 0;
  __syncthreads();

  // grad_out rows of NC 16-byte chunks; chunk k of unit u is stored at
  // position k ^ swz(u) of its row, so that the first chunks of rows read by
  // lanes with unrelated units spread over all eight 16-byte bank groups
  constexpr int NC = NW / 4;
  constexpr int kSwzShift = NC == 1 ? 0 : NC == 2 ? 2 : 1;
  auto swz = [](int u) { return (u >> kSwzShift) & (NC - 1); };
  if (local < nunit) {
    uint4* dst = reinterpret_cast<uint4*>(gos + local * NW);
#pragma unroll
    for (int k = 0; k < NC; ++k)
      dst[k ^ swz(local)] = make_uint4(gw[4 * k], gw[4 * k + 1], gw[4 * k + 2], gw[4 * k + 3]);
  }
  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) {
    mx = -INFINITY;
    for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(mrow + p));
    float s = 0.f;
    for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(mrow + p) - mx);
    inv = 1.f / s;
  }

  // per point: (rank << 16) | cell for an in-window sample, else -1, and its
  // weights; far samples are marked in a bit mask and done after the loop
  int code[KPN];
  Wq wq[KPN];
  uint32_t far = 0;
#pragma unroll(KP > 0 ? KP : 1)
  for (int p = 0; p < P; ++p) {
    code[p] = -1;
    if (!active) continue;
    float m = mm[p];
    if (kp.softmax) m = expf(m - mx) * inv;
    const float2 d = dd[p];
    const float x = location(d.x, kp.tap_x[p], scale, ref_x);
    const float y = location(d.y, kp.tap_y[p], scale, ref_y);
    if (!in_box(x, y, W, H)) continue;
    const float xf = floorf(x), yf = floorf(y);
    const int x0 = (int)xf, y0 = (int)yf;
    const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
    const float w[4] = {gy * gx * m, gy * fx * m, fy * gx * m, fy * fx * m};
    const int cy = y0 - wy0, cx = x0 - wx0;
    if ((unsigned)cy < (unsigned)(wg.WH - 1) && (unsigned)cx < (unsigned)cw) {
      const int cell = cy * cw + cx;
      if (!DCN_IN_SPAN(count + cell, sizeof(int), count, ncell * sizeof(int), kBadShared)) {
        far |= 1u << p;
        continue;
      }
      code[p] = (atomicAdd(&count[cell], 1) << 16) | cell;
      if constexpr (k16) {
        wq[p].x = (uint32_t)Fma<T>::weight(w[0]) | ((uint32_t)Fma<T>::weight(w[1]) << 16);
        wq[p].y = (uint32_t)Fma<T>::weight(w[2]) | ((uint32_t)Fma<T>::weight(w[3]) << 16);
      } else {
        wq[p] = make_float4(w[0], w[1], w[2], w[3]);
      }
    } else {
      far |= 1u << p;
    }
  }
  __syncthreads();

  // ---- pass 2: list heads (block-wide exclusive scan), then each sample to
  // head + rank ----------------------------------------------------------------
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (ncell + blockDim.x - 1) / blockDim.x;
    const int b = min((int)threadIdx.x * per, ncell), e = min(b + per, ncell);
    int s = 0;
    for (int i = b; i < e; ++i) s += count[i];
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    int run = before + incl - s;
    for (int i = b; i < e; ++i) {
      head[i] = run;
      run += count[i];
    }
    if (threadIdx.x == blockDim.x - 1) head[ncell] = run;
  }
  __syncthreads();
#pragma unroll(KP > 0 ? KP : 1)
  for (int p = 0; p < P; ++p) {
    if (code[p] < 0) continue;
    const int o = head[code[p] & 0xffff] + (code[p] >> 16);
    if (!DCN_IN_SPAN(eu + o, 2, eu, nsamp * 2, kBadShared)) continue;
    if constexpr (k16) {
      wa[o] = wq[p].y;
      wb[o] = wq[p].x;
    } else {
      wa[o] = make_float2(wq[p].z, wq[p].w);
      wb[o] = make_float2(wq[p].x, wq[p].y);
    }
    eu[o] = (unsigned short)local;
  }
  __syncthreads();

  // ---- pass 3: per window pixel inside the image --------------------------
  // Warps take 32 consecutive pixels of the window (clipped to the image).
  // Afterwards each group of L = gc/4 lanes transposes its float4 chunks, so
  // that the group's lanes reduce the L chunks of one pixel side by side:
  // one vector reduction instruction then covers 32/L pixels' contiguous
  // slices instead of 32 scattered 16-byte pieces.
  constexpr int L = CPT / 4;
  const int lane = threadIdx.x & 31;
  const int ry0 = max(0, -wy0), ry1 = min(wg.WH, H - wy0);
  const int rx0 = max(0, -wx0), rx1 = min(wg.WW, W - wx0);
  const int cols = rx1 - rx0, rows = ry1 - ry0;
  const int npix = cols > 0 && rows > 0 ? rows * cols : 0;
  // A warp's consecutive pixels run along the region's longer side: visit
  // counts fall off across the halo, and a line along the long side crosses
  // fewer halo pixels (FlashInternImage-T stage 2's 43 x 22 windows: backward
  // 164 -> 150 us against rows first).
  const bool by_rows = cols >= rows;
  const int line = by_rows ? cols : rows;
  for (int base = threadIdx.x - lane; base < npix; base += blockDim.x) {
    const int i = base + lane;
    const bool valid = i < npix;
    const int across = valid ? i / line : 0, along = valid ? i - across * line : 0;
    const int ry = ry0 + (by_rows ? across : along), rx = rx0 + (by_rows ? along : across);
    const int yy = wy0 + ry, xx = wx0 + rx;
    // the cells (cy, rx - 1) and (cy, rx) of cell rows cy = ry - 1 (range a,
    // the pixel is their lower corner) and cy = ry (range b, upper corner):
    // [s, mid) lists cell rx - 1 (the pixel is its right corner), [mid, e)
    // cell rx; cells outside the window's grid are empty
    int sa = 0, ma = 0, ea = 0, sb = 0, mb = 0, eb = 0;
    const int lo = max(rx - 1, 0), hi = min(rx + 1, cw);
    if (valid && ry >= 1) {
      const int cb = (ry - 1) * cw;
      sa = head[cb + lo];
      ma = head[cb + rx];
      ea = head[cb + hi];
    }
    if (valid && ry < wg.WH - 1) {
      const int cb = ry * cw;
      sb = head[cb + lo];
      mb = head[cb + rx];
      eb = head[cb + hi];
    }
    const int na = ea - sa, nv = na + (eb - sb);
    float acc[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) acc[k] = 0.f;
    // the weight of visit v for this pixel, and the visit's unit
    auto weight = [&](int v, int& un) -> typename Fma<T>::W {
      const bool in_a = v < na;
      int o = in_a ? sa + v : sb + (v - na);
      const bool right = o < (in_a ? ma : mb);
      if (!DCN_IN_SPAN(eu + o, 2, eu, nsamp * 2, kBadShared)) o = 0;  // (checked build)
      const Wh h = (in_a ? wa : wb)[o];
      un = eu[o];
      // the right corner (x1) of the row: the high half, or .y
      if constexpr (k16) {
        return (unsigned short)(right ? h >> 16 : h & 0xffffu);
      } else {
        return right ? h.y : h.x;
      }
    };
    auto row = [&](int un, uint32_t (&vv)[NW]) {
      if (!DCN_IN_SPAN(gos + un * NW, NW * 4, gos, nunit * NW * 4, kBadShared)) un = 0;
      const uint4* src = reinterpret_cast<const uint4*>(gos + un * NW);
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const uint4 u = src[k ^ swz(un)];
        vv[4 * k] = u.x;
        vv[4 * k + 1] = u.y;
        vv[4 * k + 2] = u.z;
        vv[4 * k + 3] = u.w;
      }
    };
    // two visits per step, so that two entry -> row load chains are in flight
    int v = 0;
    for (; v + 1 < nv; v += 2) {
      int u0, u1;
      const auto w0 = weight(v, u0);
      const auto w1 = weight(v + 1, u1);
      uint32_t r0[NW], r1[NW];
      row(u0, r0);
      row(u1, r1);
      fma_words<T, NW>(acc, r0, w0);
      fma_words<T, NW>(acc, r1, w1);
    }
    if (v < nv) {
      int u0;
      const auto w0 = weight(v, u0);
      uint32_t r0[NW];
      row(u0, r0);
      fma_words<T, NW>(acc, r0, w0);
    }
    // lane j of a group holds chunks 0..L-1 of its own pixel; after the
    // transpose it holds chunk j of the group's pixels 0..L-1
    const int j = lane & (L - 1);
#pragma unroll
    for (int sb2 = 1; sb2 < L; sb2 <<= 1) {
#pragma unroll
      for (int t = 0; t < L; ++t) {
        if (t & sb2) continue;
        const bool hi_lane = (j & sb2) != 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float send = hi_lane ? acc[4 * t + e] : acc[4 * (t | sb2) + e];
          const float got = __shfl_xor_sync(0xffffffffu, send, sb2);
          if (hi_lane)
            acc[4 * t + e] = got;
          else
            acc[4 * (t | sb2) + e] = got;
        }
      }
    }
    const int pix_off = valid ? yy * W + xx : 0;
    const int g0 = lane & ~(L - 1);
    if (wg.direct) {
      // this block alone sums the plane's pixels: every pixel of the image
      // written once, in the storage type, zeros included
      const unsigned live = __ballot_sync(0xffffffffu, valid);
#pragma unroll
      for (int r = 0; r < L; ++r) {
        const int off = __shfl_sync(0xffffffffu, pix_off, g0 + r);
        if (!((live >> (g0 + r)) & 1u)) continue;
        T* dst = gdirect + img_off + (size_t)off * kp.C + 4 * j;
        if (!DCN_IN_SPAN(dst, 4 * sizeof(T), gdirect, input_bytes<T>(kp), kBadStore)) continue;
        float q[4] = {acc[4 * r], acc[4 * r + 1], acc[4 * r + 2], acc[4 * r + 3]};
        Slice<T, 4>::store(dst, q);
      }
    } else {
      const unsigned got_any = __ballot_sync(0xffffffffu, nv > 0);
#pragma unroll
      for (int r = 0; r < L; ++r) {
        const int off = __shfl_sync(0xffffffffu, pix_off, g0 + r);
        if (!((got_any >> (g0 + r)) & 1u)) continue;
        float* dst = gin + img_off + (size_t)off * kp.C + 4 * j;
        if (!DCN_IN_SPAN(dst, 16, gin, gin_bytes, kBadScatter)) continue;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(acc[4 * r]),
                     "f"(acc[4 * r + 1]), "f"(acc[4 * r + 2]), "f"(acc[4 * r + 3]));
      }
    }
  }
  // far samples (rare): the point again, its four corners straight to memory.
  // Done last, so that no barrier of the passes above waits for these
  // reductions.
  if (far) {
    if (kp.softmax) {
      mx = -INFINITY;
      for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(mrow + p));
      float s = 0.f;
      for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(mrow + p) - mx);
      inv = 1.f / s;
    }
    while (far) {
      const int p = __ffs(far) - 1;
      far &= far - 1;
      float m = Dt<T>::one(mrow + p);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float2 d = Dt<T>::two(orow + 2 * p);
      const float x = location(d.x, kp.tap_x[p], scale, ref_x);
      const float y = location(d.y, kp.tap_y[p], scale, ref_y);
      const float xf = floorf(x), yf = floorf(y);
      const int x0 = (int)xf, y0 = (int)yf;
      const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
      const float w[4] = {gy * gx * m, gy * fx * m, fy * gx * m, fy * fx * m};
      const uint4* src = reinterpret_cast<const uint4*>(gos + local * NW);
      float gof[CPT];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 u = src[c ^ swz(local)];
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) Dt<T>::unpack(wd[i], gof + (4 * c + i) * Dt<T>::kPerWord);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int yy = y0 + (c >> 1), xx = x0 + (c & 1);
        if ((unsigned)yy >= (unsigned)H || (unsigned)xx >= (unsigned)W) continue;
        float* dst = gin + img_off + ((size_t)yy * W + xx) * kp.C;
        if (!DCN_IN_SPAN(dst, CPT * sizeof(float), gin, gin_bytes, kBadScatter)) continue;
#pragma unroll
        for (int i = 0; i < CPT; i += 4)
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i),
                       "f"(w[c] * gof[i]), "f"(w[c] * gof[i + 1]), "f"(w[c] * gof[i + 2]),
                       "f"(w[c] * gof[i + 3]));
      }
    }
  }
}

template <typename T, int NW, int KP>
__global__ void __launch_bounds__(256, NW <= 8 ? 3 : 2)
bwd_input_kernel(const KParams kp, const WinGeom wg, const T* __restrict__ gout,
                 const T* __restrict__ offset, const T* __restrict__ mask,
                 float* __restrict__ gin, T* __restrict__ gdirect) {
  input_block<T, NW, KP>(kp, wg, gout, offset, mask, gin, gdirect, blockIdx.x);
}

// Both halves in one launch: their blocks interleaved one to one (then the
// rest of the longer list), so that every SM runs gather-bound sample blocks
// and shared-memory-bound input blocks side by side instead of one kind after
// the other.  The two halves share no data: the sample half writes grad_offset
// and grad_mask, the input half reduces into the cleared accumulator.
template <typename T, int CPT, int NW, int KP>
__global__ void __launch_bounds__(256, 3)
bwd_both_kernel(const KParams kp, const WinGeom wg, const T* __restrict__ gout,
                const T* __restrict__ input, const T* __restrict__ offset,
                const T* __restrict__ mask, T* __restrict__ goff, T* __restrict__ gmask, int la,
                int lb, float* __restrict__ gin, T* __restrict__ gdirect, unsigned n_sample,
                unsigned n_input) {
  const unsigned b = blockIdx.x, m = min(n_sample, n_input);
  bool sample;
  unsigned id;
  if (b < 2 * m) {
    sample = (b & 1) == 0;
    id = b >> 1;
  } else {
    sample = n_sample > n_input;
    id = b - m;
  }
  if (sample)
    sample_block<T, CPT, KP>(kp, gout, input, offset, mask, goff, gmask, la, lb, id);
  else
    input_block<T, NW, KP>(kp, wg, gout, offset, mask, gin, gdirect, id);
}


// ---- launches ----------------------------------------------------------------

template <typename T, int CPT>
static cudaError_t launch_sample_t(const KParams& kp, const T* go_, const T* i_, const T* o_,
                                   const T* m_, T* goff_, T* gm_, int la, int lb,
                                   cudaStream_t s) {
  constexpr int bytes = CPT * (int)sizeof(T);
  if constexpr (bytes >= 16 && bytes <= 64) {
    const int chunks = kp.gc / CPT;
    const int block = 256;
    const long long grid = kp.tile_w > 0 ? (long long)kp.N * kp.tiles_w * kp.tiles_h
                                         : (kp.units * chunks + block - 1) / block;
    if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
    const size_t smem =
        la > 0 ? (size_t)(block / chunks) * (stage_stride(la, sizeof(T)) + lb) * sizeof(T) : 0;
    auto k9 = bwd_sample_kernel<T, CPT, 9>;
    auto k8 = bwd_sample_kernel<T, CPT, 8>;
    auto k0 = bwd_sample_kernel<T, CPT, 0>;
    auto k = kp.P == 9 ? k9 : kp.P == 8 ? k8 : k0;
    if (smem > 48 * 1024) {
      cudaError_t e =
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    k<<<(unsigned)grid, block, smem, s>>>(kp, go_, i_, o_, m_, goff_, gm_, la, lb);
    return cudaGetLastError();
  } else {
    return cudaErrorInvalidValue;
  }
}

template <typename T, int NW>
static cudaError_t launch_input_t(const KParams& kp, const WinGeom& wg, const T* go_,
                                  const T* o_, const T* m_, float* acc, T* gin_, cudaStream_t s) {
  const size_t smem = split_smem_bytes(wg, kp.P, kp.gc, (int)sizeof(T));
  auto k9 = bwd_input_kernel<T, NW, 9>;
  auto k8 = bwd_input_kernel<T, NW, 8>;
  auto k0 = bwd_input_kernel<T, NW, 0>;
  auto k = kp.P == 9 ? k9 : kp.P == 8 ? k8 : k0;
  // shared memory before L1: this kernel reads nothing twice from memory
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const long long blocks = (long long)kp.N * kp.G * wg.tiles_h * wg.tiles_w;
  if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
  k<<<(unsigned)blocks, 256, smem, s>>>(kp, wg, go_, o_, m_, acc, gin_);
  return cudaGetLastError();
}

// Both halves as one launch of bwd_both_kernel (the bwd_fuse switch at 0: two launches).
template <typename T, int CPT, int NW>
static cudaError_t launch_both_t(const KParams& kp, const WinGeom& wg, const T* go_, const T* i_,
                                 const T* o_, const T* m_, T* goff_, T* gm_, int la, int lb,
                                 float* acc, T* gin_, cudaStream_t s) {
  const int chunks = kp.gc / CPT;
  const int block = 256;
  const long long na = kp.tile_w > 0 ? (long long)kp.N * kp.tiles_w * kp.tiles_h
                                     : (kp.units * chunks + block - 1) / block;
  const long long nb = (long long)kp.N * kp.G * wg.tiles_h * wg.tiles_w;
  if (na + nb > INT_MAX) return cudaErrorInvalidConfiguration;
  const size_t sa =
      la > 0 ? (size_t)(block / chunks) * (stage_stride(la, sizeof(T)) + lb) * sizeof(T) : 0;
  const size_t sb = split_smem_bytes(wg, kp.P, kp.gc, (int)sizeof(T));
  const size_t smem = sa > sb ? sa : sb;
  auto k = kp.P == 9 ? bwd_both_kernel<T, CPT, NW, 9>
         : kp.P == 8 ? bwd_both_kernel<T, CPT, NW, 8>
                     : bwd_both_kernel<T, CPT, NW, 0>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k<<<(unsigned)(na + nb), block, smem, s>>>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc,
                                             gin_, (unsigned)na, (unsigned)nb);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_split(const KParams& kp, const WinGeom& wg, int cpt, int la, int lb,
                                const void* gout, const void* in, const void* off, const void* msk,
                                float* acc, void* gin, void* goff, void* gmask, cudaStream_t s) {
  const T* go_ = static_cast<const T*>(gout);
  const T* i_ = static_cast<const T*>(in);
  const T* o_ = static_cast<const T*>(off);
  const T* m_ = static_cast<const T*>(msk);
  T* goff_ = static_cast<T*>(goff);
  T* gm_ = static_cast<T*>(gmask);
  T* gin_ = static_cast<T*>(gin);
  cudaError_t e;
  const int nw = kp.gc * (int)sizeof(T) / 4;
  if (options().bwd_fuse) {
    // the (channels per sample thread, words per unit row) pairs that occur
    if constexpr (sizeof(T) == 2) {
      if (cpt == 8 && nw == 4)
        e = launch_both_t<T, 8, 4>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else if (cpt == 16 && nw == 8)
        e = launch_both_t<T, 16, 8>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else if (cpt == 16 && nw == 16)
        e = launch_both_t<T, 16, 16>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else
        return cudaErrorInvalidValue;
    } else {
      if (cpt == 4 && nw == 4)
        e = launch_both_t<T, 4, 4>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else if (cpt == 8 && nw == 8)
        e = launch_both_t<T, 8, 8>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else if (cpt == 16 && nw == 16)
        e = launch_both_t<T, 16, 16>(kp, wg, go_, i_, o_, m_, goff_, gm_, la, lb, acc, gin_, s);
      else
        return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if ((void*)acc != gin && !wg.direct) {
      const int dt = std::is_same<T, __half>::value ? DCN_F16 : DCN_BF16;
      return launch_round(dt, acc, gin, (long long)kp.N * kp.H * kp.W * kp.C, s);
    }
    return cudaSuccess;
  }
  switch (cpt) {
    case 4: e = launch_sample_t<T, 4>(kp, go_, i_, o_, m_, goff_, gm_, la, lb, s); break;
    case 8: e = launch_sample_t<T, 8>(kp, go_, i_, o_, m_, goff_, gm_, la, lb, s); break;
    case 16: e = launch_sample_t<T, 16>(kp, go_, i_, o_, m_, goff_, gm_, la, lb, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  switch (nw) {
    case 4: e = launch_input_t<T, 4>(kp, wg, go_, o_, m_, acc, gin_, s); break;
    case 8: e = launch_input_t<T, 8>(kp, wg, go_, o_, m_, acc, gin_, s); break;
    case 16: e = launch_input_t<T, 16>(kp, wg, go_, o_, m_, acc, gin_, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if ((void*)acc != gin && !wg.direct) {
    const int dt = std::is_same<T, __half>::value ? DCN_F16 : DCN_BF16;
    return launch_round(dt, acc, gin, (long long)kp.N * kp.H * kp.W * kp.C, s);
  }
  return cudaSuccess;
}

cudaError_t launch_bwd_split(const KParams& kp, const WinGeom& wg, int dtype, int cpt, int la,
                             int lb, const void* gout, const void* in, const void* off,
                             const void* msk, float* gin_acc, void* gin, void* goff, void* gmask,
                             cudaStream_t s) {
  switch (dtype) {
    case DCN_F32:
      return launch_split<float>(kp, wg, cpt, la, lb, gout, in, off, msk, gin_acc, gin, goff,
                                 gmask, s);
    case DCN_F16:
      return launch_split<__half>(kp, wg, cpt, la, lb, gout, in, off, msk, gin_acc, gin, goff,
                                  gmask, s);
    case DCN_BF16:
      return launch_split<__nv_bfloat16>(kp, wg, cpt, la, lb, gout, in, off, msk, gin_acc, gin,
                                         goff, gmask, s);
    default: return cudaErrorInvalidValue;
  }
}

DCN_BOUNDS_READER(bwd_split)

}  // namespace dcn
