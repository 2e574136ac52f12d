// dcn_bwd_window.cu -- the backward with grad_input summed on chip.
//
// grad_input is the transpose of the forward's gather: input pixel q receives
// m * w_k(q) * grad_out[u] from every sample (u, p) whose bilinear cell has q
// as corner k.  Scattering that straight from the samples costs one float32
// reduction into L2 per (sample, corner, channel slice), and L2 reductions are
// what limits a scattering backward on this GPU.  Here a CTA owns TH x TW
// output pixels of one (image, group) and a window of input pixels around
// their footprint, and works in three passes:
//
//   1. one thread per (output pixel, channel slice), like the forward: the
//      sampling locations, the four corners, dk = sum_c grad_out_c *
//      corner_k,c reduced over the unit's lanes, grad_offset and grad_mask
//      (through the softmax Jacobian for DCNv3).  Each sample whose bilinear
//      cell lies inside the window is counted in its cell with a
//      shared-memory integer atomic after the point loop; samples whose cell
//      leaves the window ("far", rare) are added to global memory there.
//   2. a counting sort by cell: each unit recomputes its in-window samples'
//      fractions and weights into their cell's slots (with its output pixel's
//      index in the tile).
//   3. one thread per (window pixel, channel slice): the sum of m * w *
//      grad_out over the four cells that have the pixel as a corner, in
//      float32 registers, with grad_out read from shared memory where pass 1
//      left it; then one vector reduction per four channels into the float32
//      accumulator, only for pixels that received something.
//
// Windows of neighbouring CTAs overlap, so the accumulator is cleared before
// the launch and reduced into.  No shared-memory float atomics are used.
#include <climits>
#include <type_traits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {

template <typename T>
__device__ __forceinline__ void softmax_stats_w(const T* row, int P, float& mx, float& inv) {
  mx = -INFINITY;
  for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(row + p));
  float s = 0.f;
  for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(row + p) - mx);
  inv = 1.f / s;
}

template <typename T, int CPT, int KP>
__global__ void __launch_bounds__(256, 3)
bwd_window_kernel(const KParams kp, const WinGeom wg, const T* __restrict__ gout,
                  const T* __restrict__ input, const T* __restrict__ offset,
                  const T* __restrict__ mask, float* __restrict__ gin, T* __restrict__ goff,
                  T* __restrict__ gmask) {
  constexpr int NW = CPT * (int)sizeof(T) / 4;
  extern __shared__ __align__(16) unsigned char smem[];
  const int P = KP > 0 ? KP : kp.P;
  const int chunks = kp.gc / CPT;
  const int nunit = wg.TH * wg.TW;
  const int nsamp = nunit * P;
  const int cw = wg.WW - 1, ncell = (wg.WH - 1) * cw;
  const int gwords = kp.gc * (int)sizeof(T) / 4;            // grad_out words per unit
  float4* sorted = reinterpret_cast<float4*>(smem);             // nsamp: fx, fy, m, pixel
  uint32_t* gos = reinterpret_cast<uint32_t*>(sorted + nsamp);  // nunit * gwords
  int* count = reinterpret_cast<int*>(gos + nunit * gwords);    // ncell
  int* head = count + ncell;                                    // ncell + 1
  int* cursor = head + ncell + 1;                               // ncell

  const int tiles = wg.tiles_h * wg.tiles_w;
  const int ng = blockIdx.x / tiles, t = blockIdx.x - ng * tiles;
  const int n = ng / kp.G, g = ng - n * kp.G;
  const int th = t / wg.tiles_w, tw = t - th * wg.tiles_w;
  const int ho0 = th * wg.TH, wo0 = tw * wg.TW;
  const int wy0 = ho0 * kp.stride_h + wg.org_y, wx0 = wo0 * kp.stride_w + wg.org_x;

  for (int i = threadIdx.x; i < ncell; i += blockDim.x) count[i] = 0;
  __syncthreads();

  // ---- pass 1: per (output pixel, slice) ------------------------------------
  const int local = threadIdx.x / chunks, slice = threadIdx.x - local * chunks;
  const int lh = local / wg.TW, lw = local - lh * wg.TW;
  const int ho = ho0 + lh, wo = wo0 + lw;
  const bool active = local < nunit && ho < kp.Ho && wo < kp.Wo;
  const bool leader = active && slice == 0;
  const int c0 = slice * CPT;
  const long long unit =
      active ? (((long long)n * kp.Ho + ho) * kp.Wo + wo) * kp.G + g : 0;
  const T* mrow = mask + unit * kp.os_mask;
  const T* orow = offset + unit * kp.os_off;
  const size_t img_off = (size_t)n * kp.H * kp.W * kp.C + g * kp.gc + c0;
  const T* img = input + img_off;
  const uint32_t W = kp.W, H = kp.H, C = kp.C, WC = (uint32_t)kp.W * kp.C;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  uint32_t gw[NW];
  if (active) {
    ldg_words<NW>(gout + unit * kp.gc + c0, gw);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) gw[i] = 0u;
  }
  if (local < nunit) {
#pragma unroll
    for (int i = 0; i < NW; ++i) gos[local * gwords + slice * NW + i] = gw[i];
  }
  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) softmax_stats_w(mrow, P, mx, inv);

  float gm_row[KP > 0 ? KP : 16];
  int code[KP > 0 ? KP : 16];  // per point: window cell, -1 no sample, -2 far sample
  float dot = 0.f;

#pragma unroll(KP > 0 ? KP : 1)
  for (int p = 0; p < P; ++p) {
    float m = 0.f, x = -4.f, y = -4.f;
    if (active) {
      m = Dt<T>::one(mrow + p);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float2 d = Dt<T>::two(orow + 2 * p);
      x = location(d.x, kp.tap_x[p], scale, ref_x);
      y = location(d.y, kp.tap_y[p], scale, ref_y);
    }
    const bool valid = active && in_box(x, y, kp.W, kp.H);
    if (!valid) {
      x = -4.f;
      y = -4.f;
    }
    const float xf = floorf(x), yf = floorf(y);
    const int x0 = (int)xf, y0 = (int)yf;
    const float fx = x - xf, fy = y - yf;
    const bool vx0 = (uint32_t)x0 < W, vx1 = (uint32_t)(x0 + 1) < W;
    const bool vy0 = (uint32_t)y0 < H, vy1 = (uint32_t)(y0 + 1) < H;
    const uint32_t xa = min((uint32_t)x0, W - 1), xb = min((uint32_t)(x0 + 1), W - 1);
    const uint32_t ya = min((uint32_t)y0, H - 1), yb = min((uint32_t)(y0 + 1), H - 1);
    const uint32_t off[4] = {ya * WC + xa * C, ya * WC + xb * C, yb * WC + xa * C,
                             yb * WC + xb * C};
    const bool ok[4] = {vy0 && vx0, vy0 && vx1, vy1 && vx0, vy1 && vx1};
    float dk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t v[NW];
      ldg_words<NW>(img + off[k], v);
      float s[2] = {0.f, 0.f};  // sum_c grad_out_c * corner_c
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < NW; ++i) dot_word<T>(s[0], s[1], v[i], gw[i]);
      } else {
#pragma unroll
        for (int i = 0; i < NW; ++i)
          s[i & 1] = fmaf(__uint_as_float(gw[i]), __uint_as_float(v[i]), s[i & 1]);
      }
      dk[k] = ok[k] ? s[0] + s[1] : 0.f;
    }
    // the sample's cell relative to the window (-2: outside it, "far")
    const int cy = y0 - wy0, cx = x0 - wx0;
    const bool inwin = (unsigned)cy < (unsigned)(wg.WH - 1) && (unsigned)cx < (unsigned)cw;
    code[p] = !valid ? -1 : inwin ? cy * cw + cx : -2;
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
      T* go2 = goff + unit * kp.os_off + p * 2;
      go2[0] = Dt<T>::from_f(gox);
      go2[1] = Dt<T>::from_f(goy);
      if (kp.softmax) {
        gm_row[p] = gm;
        dot = fmaf(m, gm, dot);
      } else {
        gmask[unit * kp.os_mask + p] = Dt<T>::from_f(gm);
      }
    }
  }
  if (leader && kp.softmax) {
    for (int p = 0; p < P; ++p) {
      const float m = expf(Dt<T>::one(mrow + p) - mx) * inv;
      gmask[unit * kp.os_mask + p] = Dt<T>::from_f(m * (gm_row[p] - dot));
    }
  }
  if (leader && kp.merged)
    for (int i = 3 * P; i < kp.os_off; ++i) goff[unit * kp.os_off + i] = Dt<T>::from_f(0.f);
  // per-cell counts, and the far samples' share of grad_input straight to memory
  if (active) {
    for (int p = 0; p < P; ++p) {
      const int cell = code[p];
      if (cell >= 0) {
        if (slice == 0) atomicAdd(&count[cell], 1);
      } else if (cell == -2) {
        float m = Dt<T>::one(mrow + p);
        if (kp.softmax) m = expf(m - mx) * inv;
        const float2 d = Dt<T>::two(orow + 2 * p);
        const float x = location(d.x, kp.tap_x[p], scale, ref_x);
        const float y = location(d.y, kp.tap_y[p], scale, ref_y);
        const float xf = floorf(x), yf = floorf(y);
        const int x0 = (int)xf, y0 = (int)yf;
        const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
        const float w[4] = {gy * gx * m, gy * fx * m, fy * gx * m, fy * fx * m};
        float gof[CPT];
#pragma unroll
        for (int i = 0; i < NW; ++i) Dt<T>::unpack(gw[i], gof + i * Dt<T>::kPerWord);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int yy = y0 + (k >> 1), xx = x0 + (k & 1);
          if ((unsigned)yy >= H || (unsigned)xx >= W) continue;
          float* dst = gin + img_off + (uint32_t)yy * WC + (uint32_t)xx * C;
#pragma unroll
          for (int i = 0; i < CPT; i += 4)
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i),
                         "f"(w[k] * gof[i]), "f"(w[k] * gof[i + 1]), "f"(w[k] * gof[i + 2]),
                         "f"(w[k] * gof[i + 3]));
        }
      }
    }
  }
  __syncthreads();

  // ---- pass 2: counting sort of the entries by cell ---------------------------
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (ncell + 31) / 32;
    const int b = min(lane * per, ncell), e = min(b + per, ncell);
    int s = 0;
    for (int i = b; i < e; ++i) s += count[i];
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - s;
    for (int i = b; i < e; ++i) {
      head[i] = run;
      cursor[i] = run;
      run += count[i];
    }
    if (lane == 31) head[ncell] = incl;
  }
  __syncthreads();
  // each unit's in-window samples, recomputed, into their cell's slots
  if (leader) {
    for (int p = 0; p < P; ++p) {
      const int cell = code[p];
      if (cell < 0) continue;
      float m = Dt<T>::one(mrow + p);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float2 d = Dt<T>::two(orow + 2 * p);
      const float x = location(d.x, kp.tap_x[p], scale, ref_x);
      const float y = location(d.y, kp.tap_y[p], scale, ref_y);
      const int o = atomicAdd(&cursor[cell], 1);
      sorted[o] = make_float4(x - floorf(x), y - floorf(y), m, __int_as_float(local));
    }
  }
  __syncthreads();

  // ---- pass 3: per (window pixel, slice): sum, then one reduction ------------
  const int npix = wg.WH * wg.WW;
  for (int i = threadIdx.x; i < npix * chunks; i += blockDim.x) {
    const int pix = i / chunks, sl = i - pix * chunks;
    const int ry = pix / wg.WW, rx = pix - ry * wg.WW;
    const int yy = wy0 + ry, xx = wx0 + rx;
    if ((unsigned)yy >= H || (unsigned)xx >= W) continue;
    float acc[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) acc[k] = 0.f;
    bool any = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int cy = ry - 1 + (q >> 1), cx = rx - 1 + (q & 1);
      if ((unsigned)cy >= (unsigned)(wg.WH - 1) || (unsigned)cx >= (unsigned)cw) continue;
      const int cell = cy * cw + cx;
      const bool lower_y = (q >> 1) == 0, lower_x = (q & 1) == 0;  // pixel is the cell's +1 corner
      for (int o = head[cell]; o < head[cell + 1]; ++o) {
        const float4 e = sorted[o];
        const float w = (lower_y ? e.y : 1.f - e.y) * (lower_x ? e.x : 1.f - e.x) * e.z;
        const uint32_t* src = gos + __float_as_int(e.w) * gwords + sl * NW;
        uint32_t v[NW];
#pragma unroll
        for (int k = 0; k < NW; k += 4) {
          const uint4 u = *reinterpret_cast<const uint4*>(src + k);
          v[k] = u.x; v[k + 1] = u.y; v[k + 2] = u.z; v[k + 3] = u.w;
        }
        fma_words<T, NW>(acc, v, Fma<T>::weight(w));
        any = true;
      }
    }
    if (!any) continue;
    float* dst = gin + (((size_t)n * kp.H + yy) * kp.W + xx) * kp.C + g * kp.gc + sl * CPT;
#pragma unroll
    for (int k = 0; k < CPT; k += 4)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + k), "f"(acc[k]),
                   "f"(acc[k + 1]), "f"(acc[k + 2]), "f"(acc[k + 3]));
  }
}

template <typename T, int CPT>
static cudaError_t launch_window_t(const KParams& kp, const WinGeom& wg, const T* go_,
                                   const T* i_, const T* o_, const T* m_, float* acc, T* goff_,
                                   T* gm_, cudaStream_t s) {
  constexpr int bytes = CPT * (int)sizeof(T);
  if constexpr (bytes >= 16 && bytes <= 64) {
    const size_t smem = window_smem_bytes(wg, kp.P, kp.gc, (int)sizeof(T));
    auto k9 = bwd_window_kernel<T, CPT, 9>;
    auto k8 = bwd_window_kernel<T, CPT, 8>;
    auto k0 = bwd_window_kernel<T, CPT, 0>;
    auto k = kp.P == 9 ? k9 : kp.P == 8 ? k8 : k0;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
    }
    const long long blocks = (long long)kp.N * kp.G * wg.tiles_h * wg.tiles_w;
    if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
    k<<<(unsigned)blocks, 256, smem, s>>>(kp, wg, go_, i_, o_, m_, acc, goff_, gm_);
    return cudaGetLastError();
  } else {
    return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_window(const KParams& kp, const WinGeom& wg, int cpt, const void* gout,
                                 const void* in, const void* off, const void* msk, float* acc,
                                 void* gin, void* goff, void* gmask, cudaStream_t s) {
  const T* go_ = static_cast<const T*>(gout);
  const T* i_ = static_cast<const T*>(in);
  const T* o_ = static_cast<const T*>(off);
  const T* m_ = static_cast<const T*>(msk);
  T* goff_ = static_cast<T*>(goff);
  T* gm_ = static_cast<T*>(gmask);
  cudaError_t e;
  switch (cpt) {
    case 4: e = launch_window_t<T, 4>(kp, wg, go_, i_, o_, m_, acc, goff_, gm_, s); break;
    case 8: e = launch_window_t<T, 8>(kp, wg, go_, i_, o_, m_, acc, goff_, gm_, s); break;
    case 16: e = launch_window_t<T, 16>(kp, wg, go_, i_, o_, m_, acc, goff_, gm_, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if ((void*)acc != gin) {
    const int dt = std::is_same<T, __half>::value ? DCN_F16 : DCN_BF16;
    return launch_round(dt, acc, gin, (long long)kp.N * kp.H * kp.W * kp.C, s);
  }
  return cudaSuccess;
}

cudaError_t launch_bwd_window(const KParams& kp, const WinGeom& wg, int dtype, int cpt,
                              const void* gout, const void* in, const void* off, const void* msk,
                              float* gin_acc, void* gin, void* goff, void* gmask, cudaStream_t s) {
  switch (dtype) {
    case DCN_F32:
      return launch_window<float>(kp, wg, cpt, gout, in, off, msk, gin_acc, gin, goff, gmask, s);
    case DCN_F16:
      return launch_window<__half>(kp, wg, cpt, gout, in, off, msk, gin_acc, gin, goff, gmask, s);
    case DCN_BF16:
      return launch_window<__nv_bfloat16>(kp, wg, cpt, gout, in, off, msk, gin_acc, gin, goff,
                                          gmask, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dcn
