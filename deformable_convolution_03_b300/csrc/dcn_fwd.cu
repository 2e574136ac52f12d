// dcn_fwd.cu -- forward of the DCNv3 / DCNv4 core deformable aggregation.
//
// One fused pass, no intermediate in global memory: for each (pixel, group,
// channel slice) a thread forms the P sampling locations, gathers the four
// bilinear corners of its channel slice, weights them by the modulation
// weight (softmax over the points for DCNv3, computed in registers) and
// accumulates in float32.  This is the computation of dcnv3_core_pytorch on
// the page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读",
// section 四 steps 2-5, fused the way the FlashInternImage page's section 2.2
// ("Flash 式 DCNv3 内核") describes: sampling, modulation and accumulation on
// chip, nothing written back but the output.
#include <climits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {

// (n, ho, wo, g) of a unit = flat (pixel, group) index, pixels row-major.
struct Unit {
  int n, ho, wo, g;
};

__device__ __forceinline__ Unit decompose(long long unit, const KParams& kp) {
  Unit u;
  if (kp.units <= (long long)INT_MAX) {
    int q = (int)unit;
    u.g = q % kp.G;
    q /= kp.G;
    u.wo = q % kp.Wo;
    q /= kp.Wo;
    u.ho = q % kp.Ho;
    u.n = q / kp.Ho;
  } else {
    long long q = unit;
    u.g = (int)(q % kp.G);
    q /= kp.G;
    u.wo = (int)(q % kp.Wo);
    q /= kp.Wo;
    u.ho = (int)(q % kp.Ho);
    u.n = (int)(q / kp.Ho);
  }
  return u;
}

// Softmax statistics of one row of P logits: the maximum and 1/sum(exp).
template <typename T>
__device__ __forceinline__ void softmax_stats(const T* row, int P, float& mx, float& inv) {
  mx = -INFINITY;
  for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(row + p));
  float s = 0.f;
  for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(row + p) - mx);
  inv = 1.f / s;
}

template <typename T, int CPT>
__global__ void __launch_bounds__(256)
fwd_kernel(const KParams kp, const T* __restrict__ input, const T* __restrict__ offset,
           const T* __restrict__ mask, T* __restrict__ output) {
  const int chunks = kp.gc / CPT;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= kp.units * chunks) return;
  const long long unit = item / chunks;
  const int c0 = (int)(item - unit * chunks) * CPT;
  const Unit u = decompose(unit, kp);

  const T* mrow = mask + unit * kp.os_mask;
  const T* orow = offset + unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow)) return;
  float mx = 0.f, inv = 1.f;
  if (kp.softmax) softmax_stats(mrow, kp.P, mx, inv);

  const float ref_x = (float)(u.wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(u.ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const long long img = (long long)u.n * kp.H * kp.W;
  const int cbase = u.g * kp.gc + c0;

  float acc[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) acc[i] = 0.f;

#pragma unroll 1
  for (int p = 0; p < kp.P; ++p) {
    float m = Dt<T>::one(mrow + p);
    if (kp.softmax) m = expf(m - mx) * inv;
    const float2 d = Dt<T>::two(orow + 2 * p);
    const float x = location(d.x, kp.tap_x[p], kp.offset_scale, ref_x);
    const float y = location(d.y, kp.tap_y[p], kp.offset_scale, ref_y);
    if (!in_box(x, y, kp.W, kp.H)) continue;
    const float x0f = floorf(x), y0f = floorf(y);
    const int x0 = (int)x0f, y0 = (int)y0f;
    const float fx = x - x0f, fy = y - y0f;
    const float gx = 1.f - fx, gy = 1.f - fy;
    const float w[4] = {gy * gx * m, gy * fx * m, fy * gx * m, fy * fx * m};
    const bool ok[4] = {y0 >= 0 && x0 >= 0, y0 >= 0 && x0 + 1 < kp.W,
                        y0 + 1 < kp.H && x0 >= 0, y0 + 1 < kp.H && x0 + 1 < kp.W};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (!ok[k]) continue;
      const long long pix = img + (long long)(y0 + (k >> 1)) * kp.W + (x0 + (k & 1));
      float v[CPT];
      load_slice_in<T, CPT>(input + pix * kp.C + cbase, v, input, input_bytes<T>(kp));
#pragma unroll
      for (int i = 0; i < CPT; ++i) acc[i] = fmaf(w[k], v[i], acc[i]);
    }
  }
  if (out_in(kp, output, output + unit * kp.gc + c0, CPT))
    Slice<T, CPT>::store(output + unit * kp.gc + c0, acc);
}

// The wide kernel: one thread per (unit, slice of CPT channels) where a
// slice is 16, 32 or 64 bytes and every corner is one or two 256-bit loads.
// Corners outside the image keep a valid (clamped) address and get weight 0,
// so every thread runs the same straight-line code for every point.  With
// kp.tile_w > 0 a block covers a tile_w x tile_h patch of output pixels (all
// groups and slices), so that the block's samples share input lines in L1;
// otherwise it covers 256 consecutive (unit, slice) items.  Offsets and masks
// are read once and bypass L1.  Needs the unit count and each image's
// element count below 2^31.
template <typename T, int CPT, int KP>
__global__ void __launch_bounds__(256)
fwd_wide_kernel(const KParams kp, const T* __restrict__ input, const T* __restrict__ offset,
                const T* __restrict__ mask, T* __restrict__ output) {
  constexpr int NW = CPT * (int)sizeof(T) / 4;  // 32-bit words per corner
  const int chunks = kp.gc / CPT;
  uint32_t unit, n;
  int c0, g, ho, wo;
  if (kp.tile_w > 0) {
    // tid = (pixel-in-tile * G + g) * chunks + slice
    const int per_px = kp.G * chunks;
    const int lp = threadIdx.x / per_px, r = threadIdx.x - lp * per_px;
    g = r / chunks;
    c0 = (r - g * chunks) * CPT;
    const int tiles = kp.tiles_w * kp.tiles_h;
    n = blockIdx.x / tiles;
    const int t = blockIdx.x - n * tiles;
    const int ty = t / kp.tiles_w;
    ho = ty * kp.tile_h + lp / kp.tile_w;
    wo = (t - ty * kp.tiles_w) * kp.tile_w + lp % kp.tile_w;
    if (ho >= kp.Ho || wo >= kp.Wo) return;
    unit = ((n * (uint32_t)kp.Ho + ho) * kp.Wo + wo) * kp.G + g;
  } else {
    const uint32_t item = blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= (uint32_t)(kp.units * chunks)) return;
    unit = chunks == 1 ? item : item / (uint32_t)chunks;
    c0 = (int)(item - unit * chunks) * CPT;
    const uint32_t q1 = kp.div_G.div(unit);
    g = (int)(unit - q1 * (uint32_t)kp.G);
    const uint32_t q2 = kp.div_Wo.div(q1);
    wo = (int)(q1 - q2 * (uint32_t)kp.Wo);
    n = kp.div_Ho.div(q2);
    ho = (int)(q2 - n * (uint32_t)kp.Ho);
  }

  const int P = KP > 0 ? KP : kp.P;
  const T* mrow = mask + (size_t)unit * kp.os_mask;
  const T* orow = offset + (size_t)unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow) ||
      (KP == 9 && sizeof(T) == 2 && kp.merged_rows64 &&
       !DCN_IN_SPAN(orow, 64, offset, offset_bytes<T>(kp), kBadRow)))
    return;
  const T* img = input + (size_t)n * kp.H * kp.W * kp.C + g * kp.gc + c0;
  const uint32_t W = kp.W, H = kp.H, C = kp.C, WC = (uint32_t)kp.W * kp.C;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  // separate offset / mask tensors and a compile-time point count: the rows
  // with a few aligned vector loads
  UnitRows<T, KP> rows;
  bool vec = false;
  // (not for 64-byte float32 slices, whose corners already fill the registers)
  constexpr bool kVecRows = KP > 0 && (sizeof(T) == 2 || CPT <= 8);
  if constexpr (kVecRows) vec = !kp.merged && rows.load(offset, mask, kp.units, orow, mrow);

  // DCNv3: softmax statistics of the unit's logits
  float mx = 0.f, inv = 1.f;
  if (kp.softmax) {
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

  float acc[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) acc[i] = 0.f;

  // merged rows of P = 9 in 16-bit storage: the whole row in 16 registers
  constexpr bool kRow64 = KP == 9 && sizeof(T) == 2;
  uint32_t row[kRow64 ? 16 : 1];
  const bool row64 = kRow64 && kp.merged_rows64;
  if constexpr (kRow64) {
    if (row64) {
      uint32_t (&r16)[16] = *reinterpret_cast<uint32_t(*)[16]>(row);
      ldg_words<16>(orow, r16);
    }
  }

#pragma unroll(KP > 0 ? KP : 3)
  for (int p = 0; p < P; ++p) {
    float m;
    float2 d;
    if (kRow64 && row64) {
      // word p holds (dx, dy) of point p; mask p is half 18 + p
      uint32_t dw = row[kRow64 ? p : 0];
      uint32_t mw = row[kRow64 ? (18 + p) / 2 : 0];
      if constexpr (sizeof(T) == 2) {
        float lo[2], hi[2];
        Dt<T>::unpack(dw, lo);
        Dt<T>::unpack(mw, hi);
        d = make_float2(lo[0], lo[1]);
        m = hi[(18 + p) & 1];
      }
    } else if (KP > 0 && vec) {
      m = rows.msk(KP > 0 ? p : 0);
      d = rows.off(KP > 0 ? p : 0);
    } else {
      m = ld_once_1(mrow + p);
      d = ld_once_2(orow + 2 * p);
    }
    if (kp.softmax) m = expf(m - mx) * inv;
    float x = location(d.x, kp.tap_x[p], scale, ref_x);
    float y = location(d.y, kp.tap_y[p], scale, ref_y);
    if (!in_box(x, y, kp.W, kp.H)) {  // also NaN / inf: every corner falls outside
      x = -4.f;
      y = -4.f;
    }
    const float xf = floorf(x), yf = floorf(y);
    const int x0 = (int)xf, y0 = (int)yf;
    const float fx = x - xf, fy = y - yf;
    const float wy0 = (uint32_t)y0 < H ? (1.f - fy) * m : 0.f;
    const float wy1 = (uint32_t)(y0 + 1) < H ? fy * m : 0.f;
    const float wx0 = (uint32_t)x0 < W ? 1.f - fx : 0.f;
    const float wx1 = (uint32_t)(x0 + 1) < W ? fx : 0.f;
    // clamped corners: always inside the image, weight 0 when really outside
    const uint32_t xa = min((uint32_t)x0, W - 1), xb = min((uint32_t)(x0 + 1), W - 1);
    const uint32_t ya = min((uint32_t)y0, H - 1), yb = min((uint32_t)(y0 + 1), H - 1);
    const uint32_t ra = ya * WC, rb = yb * WC, ca = xa * C, cb = xb * C;
    uint32_t v00[NW], v01[NW], v10[NW], v11[NW];
    ldg_words_in<NW>(img + (ra + ca), v00, input, input_bytes<T>(kp));
    ldg_words_in<NW>(img + (ra + cb), v01, input, input_bytes<T>(kp));
    ldg_words_in<NW>(img + (rb + ca), v10, input, input_bytes<T>(kp));
    ldg_words_in<NW>(img + (rb + cb), v11, input, input_bytes<T>(kp));
    fma_words<T, NW>(acc, v00, Fma<T>::weight(wy0 * wx0));
    fma_words<T, NW>(acc, v01, Fma<T>::weight(wy0 * wx1));
    fma_words<T, NW>(acc, v10, Fma<T>::weight(wy1 * wx0));
    fma_words<T, NW>(acc, v11, Fma<T>::weight(wy1 * wx1));
  }
  if (out_in(kp, output, output + (size_t)unit * kp.gc + c0, CPT))
    Slice<T, CPT>::store(output + (size_t)unit * kp.gc + c0, acc);
}

template <typename T, int CPT>
static void launch_wide(const KParams& kp, unsigned grid, int block, cudaStream_t s, const T* i_,
                        const T* o_, const T* m_, T* y_) {
  constexpr int bytes = CPT * (int)sizeof(T);
  if constexpr (bytes >= 16 && bytes <= 64) {
    // compile-time point counts (fully unrolled) for the 3x3 kernel with and
    // without its centre; any other count takes the runtime loop
    if (kp.P == 9)
      fwd_wide_kernel<T, CPT, 9><<<grid, block, 0, s>>>(kp, i_, o_, m_, y_);
    else if (kp.P == 8)
      fwd_wide_kernel<T, CPT, 8><<<grid, block, 0, s>>>(kp, i_, o_, m_, y_);
    else
      fwd_wide_kernel<T, CPT, 0><<<grid, block, 0, s>>>(kp, i_, o_, m_, y_);
  }
}

template <typename T>
static cudaError_t launch_fwd_t(const KParams& kp, int cpt, const void* in, const void* off,
                                const void* msk, void* out, cudaStream_t s) {
  const long long items = kp.units * (kp.gc / (cpt < 0 ? -cpt : cpt));
  const int block = 256;
  const long long grid = (cpt < 0 && kp.tile_w > 0)
                             ? (long long)kp.N * kp.tiles_w * kp.tiles_h
                             : (items + block - 1) / block;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  const T* i_ = static_cast<const T*>(in);
  const T* o_ = static_cast<const T*>(off);
  const T* m_ = static_cast<const T*>(msk);
  T* y_ = static_cast<T*>(out);
  switch (cpt) {
#define DCN_CASE(K) \
    case K: fwd_kernel<T, K><<<(unsigned)grid, block, 0, s>>>(kp, i_, o_, m_, y_); break;
    DCN_CASE(1) DCN_CASE(2) DCN_CASE(4) DCN_CASE(8) DCN_CASE(16) DCN_CASE(32)
#undef DCN_CASE
    case -4: launch_wide<T, 4>(kp, (unsigned)grid, block, s, i_, o_, m_, y_); break;
    case -8: launch_wide<T, 8>(kp, (unsigned)grid, block, s, i_, o_, m_, y_); break;
    case -16: launch_wide<T, 16>(kp, (unsigned)grid, block, s, i_, o_, m_, y_); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd(const KParams& kp, int dtype, int cpt, const void* in, const void* off,
                       const void* msk, void* out, cudaStream_t s) {
  switch (dtype) {
    case DCN_F32: return launch_fwd_t<float>(kp, cpt, in, off, msk, out, s);
    case DCN_F16: return launch_fwd_t<__half>(kp, cpt, in, off, msk, out, s);
    case DCN_BF16: return launch_fwd_t<__nv_bfloat16>(kp, cpt, in, off, msk, out, s);
    default: return cudaErrorInvalidValue;
  }
}

DCN_BOUNDS_READER(fwd)

}  // namespace dcn
