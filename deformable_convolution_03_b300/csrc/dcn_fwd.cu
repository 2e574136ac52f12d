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

  const T* mrow = mask + unit * kp.P;
  const T* orow = offset + unit * kp.P * 2;
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
      Slice<T, CPT>::load(input + pix * kp.C + cbase, v);
#pragma unroll
      for (int i = 0; i < CPT; ++i) acc[i] = fmaf(w[k], v[i], acc[i]);
    }
  }
  Slice<T, CPT>::store(output + unit * kp.gc + c0, acc);
}

template <typename T>
static cudaError_t launch_fwd_t(const KParams& kp, int cpt, const void* in, const void* off,
                                const void* msk, void* out, cudaStream_t s) {
  const long long items = kp.units * (kp.gc / cpt);
  const int block = 256;
  const long long grid = (items + block - 1) / block;
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

}  // namespace dcn
