// dcn_common.cuh -- internal definitions shared by the forward and backward
// kernels of libdcn_b300: the kernel parameter record, storage-dtype traits and
// vector loads / stores of a thread's channel slice.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dcn_core.h"

namespace dcn {

// Everything a kernel needs about one call, passed by value (kernel parameter
// space, so warp-uniform reads of it are cheap).
struct KParams {
  int N, H, W, G, gc, C;     // C = G*gc
  int Ho, Wo, P;
  int stride_h, stride_w;
  int pad_h, pad_w;
  int cen_h, cen_w;          // floor(dilation*(kernel-1)/2)
  float offset_scale;
  int softmax;
  long long units;           // N*Ho*Wo*G: one (pixel, group) pair each
  // Kernel taps of the P points, in point order (x-major, centre removed when
  // asked): ix*dilation_w - cen_w and iy*dilation_h - cen_h, as floats (exact).
  float tap_x[DCN_MAX_POINTS];
  float tap_y[DCN_MAX_POINTS];
};

// ---- storage dtype traits ---------------------------------------------------

template <typename T> struct Dt;

template <> struct Dt<float> {
  static constexpr int kPerWord = 1;
  __device__ __forceinline__ static void unpack(uint32_t w, float* f) { f[0] = __uint_as_float(w); }
  __device__ __forceinline__ static uint32_t pack(const float* f) { return __float_as_uint(f[0]); }
  __device__ __forceinline__ static float one(const float* p) { return __ldg(p); }
  __device__ __forceinline__ static float2 two(const float* p) {
    return __ldg(reinterpret_cast<const float2*>(p));
  }
  __device__ __forceinline__ static float to_f(float v) { return v; }
  __device__ __forceinline__ static float from_f(float v) { return v; }
};

template <> struct Dt<__half> {
  static constexpr int kPerWord = 2;
  __device__ __forceinline__ static void unpack(uint32_t w, float* f) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 v = __half22float2(h);
    f[0] = v.x;
    f[1] = v.y;
  }
  __device__ __forceinline__ static uint32_t pack(const float* f) {
    __half2 h = __floats2half2_rn(f[0], f[1]);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static float one(const __half* p) { return __half2float(__ldg(p)); }
  __device__ __forceinline__ static float2 two(const __half* p) {
    return __half22float2(__ldg(reinterpret_cast<const __half2*>(p)));
  }
  __device__ __forceinline__ static __half from_f(float v) { return __float2half_rn(v); }
};

template <> struct Dt<__nv_bfloat16> {
  static constexpr int kPerWord = 2;
  __device__ __forceinline__ static void unpack(uint32_t w, float* f) {
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xffff0000u);
  }
  __device__ __forceinline__ static uint32_t pack(const float* f) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[0], f[1]);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static float one(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
  }
  __device__ __forceinline__ static float2 two(const __nv_bfloat16* p) {
    return __bfloat1622float2(__ldg(reinterpret_cast<const __nv_bfloat162*>(p)));
  }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// ---- a thread's slice of CPT consecutive channels ---------------------------
// The slice starts CPT*sizeof(T)-aligned (the host picks CPT so that it is),
// and is moved with the widest loads that alignment allows (16 bytes at most).

template <typename T, int CPT>
struct Slice {
  static constexpr int kBytes = CPT * (int)sizeof(T);
  static constexpr int kWords = kBytes >= 4 ? kBytes / 4 : 0;

  __device__ __forceinline__ static void load(const T* p, float (&v)[CPT]) {
    if constexpr (kBytes < 4) {
      v[0] = Dt<T>::one(p);
    } else {
      uint32_t w[kWords];
      if constexpr (kBytes % 16 == 0) {
#pragma unroll
        for (int i = 0; i < kBytes / 16; ++i) {
          uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + i);
          w[4 * i + 0] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
        }
      } else if constexpr (kBytes == 8) {
        uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = u.x; w[1] = u.y;
      } else {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
      }
#pragma unroll
      for (int i = 0; i < kWords; ++i) Dt<T>::unpack(w[i], v + i * Dt<T>::kPerWord);
    }
  }

  __device__ __forceinline__ static void store(T* p, const float (&v)[CPT]) {
    if constexpr (kBytes < 4) {
      p[0] = Dt<T>::from_f(v[0]);
    } else {
      uint32_t w[kWords];
#pragma unroll
      for (int i = 0; i < kWords; ++i) w[i] = Dt<T>::pack(v + i * Dt<T>::kPerWord);
      if constexpr (kBytes % 16 == 0) {
#pragma unroll
        for (int i = 0; i < kBytes / 16; ++i)
          reinterpret_cast<uint4*>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      } else if constexpr (kBytes == 8) {
        reinterpret_cast<uint2*>(p)[0] = make_uint2(w[0], w[1]);
      } else {
        reinterpret_cast<unsigned int*>(p)[0] = w[0];
      }
    }
  }
};

// ---- the sampling location of one point (binary32, fused multiply-adds) ------
// ref = o*stride - pad + cen (unpadded pixel units, exact in binary32);
// location = fma(offset, scale, fma(tap, scale, ref)).

__device__ __forceinline__ float location(float off, float tap, float scale, float ref) {
  return __fmaf_rn(off, scale, __fmaf_rn(tap, scale, ref));
}

// A sample contributes only when its location lies in the open box
// (-1, W) x (-1, H); NaN fails every comparison and is dropped too.
__device__ __forceinline__ bool in_box(float x, float y, int W, int H) {
  return x > -1.f && x < (float)W && y > -1.f && y < (float)H;
}

}  // namespace dcn
