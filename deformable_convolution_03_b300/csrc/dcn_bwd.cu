// dcn_bwd.cu -- backward of the DCNv3 / DCNv4 core deformable aggregation.
//
// The analytic derivative of the forward (see dcn_fwd.cu), recomputing the
// sampling locations and weights instead of saving them: the FlashInternImage
// page, section 2.2, names re-reading the saved sampling intermediates in the
// backward as the cost a fused kernel avoids, and section 5.2 that the
// backward keeps the sampling coordinates and modulation factors.  Here
// nothing but the inputs is read.
//
// Per (pixel, group, point), with v_c the bilinear sample of channel c, d_k =
// sum_c gout_c * corner_k,c over the thread's channels (reduced across the
// threads of the unit by warp shuffles):
//   dL/dm         = sum_k w_k d_k                       (w_k the bilinear weights)
//   dL/d offset_x = scale * m * (gy*(d01 - d00) + fy*(d11 - d10))
//   dL/d offset_y = scale * m * (gx*(d10 - d00) + fx*(d11 - d01))
//   dL/d input    = m * w_k * gout  scattered to each in-image corner k
//   (DCNv3)  dL/d logit_p = m_p * (dL/dm_p - sum_q m_q dL/dm_q)
// grad_input is accumulated in float32 by vector atomic adds, into the
// caller's float32 grad_input, or into a float32 workspace that a second
// kernel rounds to the storage dtype.
#include <climits>
#include <cstdlib>

#include "dcn_common.cuh"
#include "dcn_kernels.h"
#include "dcn_options.h"

namespace dcn {

struct UnitB {
  int n, ho, wo, g;
};

__device__ __forceinline__ UnitB decompose_b(long long unit, const KParams& kp) {
  UnitB u;
  long long q = unit;
  u.g = (int)(q % kp.G);
  q /= kp.G;
  u.wo = (int)(q % kp.Wo);
  q /= kp.Wo;
  u.ho = (int)(q % kp.Ho);
  u.n = (int)(q / kp.Ho);
  return u;
}

template <typename T>
__device__ __forceinline__ void softmax_stats_b(const T* row, int P, float& mx, float& inv) {
  mx = -INFINITY;
  for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(row + p));
  float s = 0.f;
  for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(row + p) - mx);
  inv = 1.f / s;
}

// Atomic float32 add of CPT consecutive values; the address is 16-byte aligned
// when CPT is a multiple of 4 and 8-byte aligned when it is even.  No kernel
// reads the accumulator it reduces into, so the reductions carry no memory
// clobber: the compiler may issue later loads ahead of them.
template <int CPT>
__device__ __forceinline__ void red_add(float* dst, const float (&v)[CPT]) {
  if constexpr (CPT % 4 == 0) {
#pragma unroll
    for (int i = 0; i < CPT; i += 4)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i), "f"(v[i]),
                   "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3]));
  } else if constexpr (CPT % 2 == 0) {
#pragma unroll
    for (int i = 0; i < CPT; i += 2)
      asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(dst + i), "f"(v[i]), "f"(v[i + 1]));
  } else {
#pragma unroll
    for (int i = 0; i < CPT; ++i) atomicAdd(dst + i, v[i]);
  }
}

// One thread per (unit, slice of CPT channels); gc/CPT is a power of two no
// larger than 32, so the threads of a unit are adjacent lanes of one warp.
// Copy n elements of T from shared to global memory with 16-byte stores when
// both ends allow it (the caller's block then writes whole sectors).
template <typename T>
__device__ __forceinline__ void block_copy_out(T* __restrict__ dst, const T* __restrict__ src,
                                               int n) {
  const int bytes = n * (int)sizeof(T);
  if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0 && (bytes & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) d4[i] = s4[i];
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
  }
}

template <typename T, int CPT>
__global__ void __launch_bounds__(256)
bwd_kernel(const KParams kp, const T* __restrict__ gout, const T* __restrict__ input,
           const T* __restrict__ offset, const T* __restrict__ mask, float* __restrict__ gin,
           T* __restrict__ goff, T* __restrict__ gmask, int stage) {
  // stage != 0: grad_offset / grad_mask rows of the block's units are put
  // together in shared memory and written out at the end with full-sector
  // stores instead of one 2- or 4-byte store per value
  extern __shared__ __align__(16) unsigned char stage_raw[];
  const int chunks = kp.gc / CPT;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool active = item < kp.units * chunks;
  const long long unit = active ? item / chunks : 0;
  const int slice = (int)(item % chunks);
  const bool leader = active && slice == 0;
  const int c0 = slice * CPT;
  const UnitB u = decompose_b(unit, kp);

  float go[CPT];
  if (active) {
    Slice<T, CPT>::load(gout + unit * kp.gc + c0, go);
  } else {
#pragma unroll
    for (int i = 0; i < CPT; ++i) go[i] = 0.f;
  }
  const T* mrow = mask + unit * kp.os_mask;
  const T* orow = offset + unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow)) {  // (checked build) read unit 0's rows
    mrow = mask;
    orow = offset;
  }
  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) softmax_stats_b(mrow, kp.P, mx, inv);

  const float ref_x = (float)(u.wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(u.ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const long long img = (long long)u.n * kp.H * kp.W;
  const int cbase = u.g * kp.gc + c0;
  const float scale = kp.offset_scale;

  float gm_row[DCN_MAX_POINTS];
  float dot = 0.f;
  T* s_off = reinterpret_cast<T*>(stage_raw);
  T* s_mask = s_off + (blockDim.x / chunks) * kp.P * 2;
  const int lunit = threadIdx.x / chunks;
  T* so_row = s_off + lunit * kp.P * 2;
  T* sm_row = s_mask + lunit * kp.P;

#pragma unroll 1
  for (int p = 0; p < kp.P; ++p) {
    float m = 0.f, x = 0.f, y = 0.f;
    if (active) {
      m = Dt<T>::one(mrow + p);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float2 d = Dt<T>::two(orow + 2 * p);
      x = location(d.x, kp.tap_x[p], scale, ref_x);
      y = location(d.y, kp.tap_y[p], scale, ref_y);
    }
    const bool valid = active && in_box(x, y, kp.W, kp.H);
    float fx = 0.f, fy = 0.f;
    float dk[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const float x0f = floorf(x), y0f = floorf(y);
      const int x0 = (int)x0f, y0 = (int)y0f;
      fx = x - x0f;
      fy = y - y0f;
      const float gx = 1.f - fx, gy = 1.f - fy;
      const float w[4] = {gy * gx * m, gy * fx * m, fy * gx * m, fy * fx * m};
      const bool ok[4] = {y0 >= 0 && x0 >= 0, y0 >= 0 && x0 + 1 < kp.W,
                          y0 + 1 < kp.H && x0 >= 0, y0 + 1 < kp.H && x0 + 1 < kp.W};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!ok[k]) continue;
        const long long pix = img + (long long)(y0 + (k >> 1)) * kp.W + (x0 + (k & 1));
        const long long at = pix * kp.C + cbase;
        float v[CPT], g[CPT];
        load_slice_in<T, CPT>(input + at, v, input, input_bytes<T>(kp));
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          s = fmaf(go[i], v[i], s);
          g[i] = w[k] * go[i];
        }
        dk[k] = s;
        if (DCN_IN_SPAN(gin + at, CPT * sizeof(float), gin, input_bytes<float>(kp), kBadScatter))
          red_add<CPT>(gin + at, g);
      }
    }
    // sum the four corner dot products over the threads of the unit
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
      T* go2 = stage ? so_row + p * 2 : goff + unit * kp.os_off + p * 2;
      go2[0] = Dt<T>::from_f(gox);
      go2[1] = Dt<T>::from_f(goy);
      if (kp.softmax) {
        gm_row[p] = gm;
        dot = fmaf(m, gm, dot);
      } else {
        (stage ? sm_row : gmask + unit * kp.os_mask)[p] = Dt<T>::from_f(gm);
      }
    }
  }
  if (leader && kp.softmax) {
    for (int p = 0; p < kp.P; ++p) {
      const float m = expf(Dt<T>::one(mrow + p) - mx) * inv;
      (stage ? sm_row : gmask + unit * kp.os_mask)[p] = Dt<T>::from_f(m * (gm_row[p] - dot));
    }
  }
  if (leader && kp.merged)
    for (int i = 3 * kp.P; i < kp.os_off; ++i) goff[unit * kp.os_off + i] = Dt<T>::from_f(0.f);
  if (stage) {
    __syncthreads();
    const int per_block = blockDim.x / chunks;
    const long long u0 = (long long)blockIdx.x * per_block;
    const int nu = (int)min((long long)per_block, kp.units - u0);
    if (nu > 0) {
      block_copy_out(goff + u0 * kp.P * 2, s_off, nu * kp.P * 2);
      block_copy_out(gmask + u0 * kp.P, s_mask, nu * kp.P);
    }
  }
}

// Any gc: one thread per unit walks all of its channels one by one.
template <typename T>
__global__ void __launch_bounds__(256)
bwd_generic_kernel(const KParams kp, const T* __restrict__ gout, const T* __restrict__ input,
                   const T* __restrict__ offset, const T* __restrict__ mask,
                   float* __restrict__ gin, T* __restrict__ goff, T* __restrict__ gmask) {
  const long long unit = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (unit >= kp.units) return;
  const UnitB u = decompose_b(unit, kp);
  const T* mrow = mask + unit * kp.os_mask;
  const T* orow = offset + unit * kp.os_off;
  const T* grow = gout + unit * kp.gc;
  if (!rows_in(kp, offset, mask, orow, mrow) || !out_in(kp, gout, grow, kp.gc)) return;
  float mx = 0.f, inv = 1.f;
  if (kp.softmax) softmax_stats_b(mrow, kp.P, mx, inv);
  const float ref_x = (float)(u.wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(u.ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const long long img = (long long)u.n * kp.H * kp.W;
  const float scale = kp.offset_scale;
  float dot = 0.f;
  for (int p = 0; p < kp.P; ++p) {
    float m = Dt<T>::one(mrow + p);
    if (kp.softmax) m = expf(m - mx) * inv;
    const float2 d = Dt<T>::two(orow + 2 * p);
    const float x = location(d.x, kp.tap_x[p], scale, ref_x);
    const float y = location(d.y, kp.tap_y[p], scale, ref_y);
    float gm = 0.f, gox = 0.f, goy = 0.f;
    if (in_box(x, y, kp.W, kp.H)) {
      const float x0f = floorf(x), y0f = floorf(y);
      const int x0 = (int)x0f, y0 = (int)y0f;
      const float fx = x - x0f, fy = y - y0f, gx = 1.f - fx, gy = 1.f - fy;
      const float w[4] = {gy * gx, gy * fx, fy * gx, fy * fx};
      const bool ok[4] = {y0 >= 0 && x0 >= 0, y0 >= 0 && x0 + 1 < kp.W,
                          y0 + 1 < kp.H && x0 >= 0, y0 + 1 < kp.H && x0 + 1 < kp.W};
      float dk[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k = 0; k < 4; ++k) {
        if (!ok[k]) continue;
        const long long pix = img + (long long)(y0 + (k >> 1)) * kp.W + (x0 + (k & 1));
        const long long at = pix * kp.C + (long long)u.g * kp.gc;
        if (!DCN_IN_SPAN(input + at, kp.gc * sizeof(T), input, input_bytes<T>(kp), kBadGather) ||
            !DCN_IN_SPAN(gin + at, kp.gc * sizeof(float), gin, input_bytes<float>(kp),
                         kBadScatter))
          continue;
        for (int c = 0; c < kp.gc; ++c) {
          const float g = Dt<T>::one(grow + c);
          dk[k] = fmaf(g, Dt<T>::one(input + at + c), dk[k]);
          atomicAdd(gin + at + c, w[k] * m * g);
        }
      }
      gm = gy * (gx * dk[0] + fx * dk[1]) + fy * (gx * dk[2] + fx * dk[3]);
      gox = scale * m * (gy * (dk[1] - dk[0]) + fy * (dk[3] - dk[2]));
      goy = scale * m * (gx * (dk[2] - dk[0]) + fx * (dk[3] - dk[1]));
    }
    T* go2 = goff + unit * kp.os_off + p * 2;
    go2[0] = Dt<T>::from_f(gox);
    go2[1] = Dt<T>::from_f(goy);
    // without softmax dL/dm is the result; with softmax it is needed again
    // after the loop, and the second pass below recomputes it.
    if (!kp.softmax) gmask[unit * kp.os_mask + p] = Dt<T>::from_f(gm);
    dot = fmaf(m, gm, dot);
  }
  if (kp.merged)
    for (int i = 3 * kp.P; i < kp.os_off; ++i) goff[unit * kp.os_off + i] = Dt<T>::from_f(0.f);
  if (!kp.softmax) return;
  // Second pass for the softmax derivative: dL/dm_p is recomputed, since a
  // per-point array would not fit in registers for large P.
  for (int p = 0; p < kp.P; ++p) {
    const float m = expf(Dt<T>::one(mrow + p) - mx) * inv;
    const float2 d = Dt<T>::two(orow + 2 * p);
    const float x = location(d.x, kp.tap_x[p], scale, ref_x);
    const float y = location(d.y, kp.tap_y[p], scale, ref_y);
    float gm = 0.f;
    if (in_box(x, y, kp.W, kp.H)) {
      const float x0f = floorf(x), y0f = floorf(y);
      const int x0 = (int)x0f, y0 = (int)y0f;
      const float fx = x - x0f, fy = y - y0f, gx = 1.f - fx, gy = 1.f - fy;
      const float w[4] = {gy * gx, gy * fx, fy * gx, fy * fx};
      const bool ok[4] = {y0 >= 0 && x0 >= 0, y0 >= 0 && x0 + 1 < kp.W,
                          y0 + 1 < kp.H && x0 >= 0, y0 + 1 < kp.H && x0 + 1 < kp.W};
      for (int k = 0; k < 4; ++k) {
        if (!ok[k]) continue;
        const long long pix = img + (long long)(y0 + (k >> 1)) * kp.W + (x0 + (k & 1));
        const long long at = pix * kp.C + (long long)u.g * kp.gc;
        if (!DCN_IN_SPAN(input + at, kp.gc * sizeof(T), input, input_bytes<T>(kp), kBadGather))
          continue;
        float s = 0.f;
        for (int c = 0; c < kp.gc; ++c)
          s = fmaf(Dt<T>::one(grow + c), Dt<T>::one(input + at + c), s);
        gm = fmaf(w[k], s, gm);
      }
    }
    gmask[unit * kp.os_mask + p] = Dt<T>::from_f(m * (gm - dot));
  }
}

// grad_input = round(float32 accumulator) in the storage dtype.
template <typename T>
__global__ void __launch_bounds__(256)
round_kernel(const float* __restrict__ acc, T* __restrict__ out, long long n) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // eight elements at a time (two 16-byte loads, one 16-byte store) when the
  // output is 16-byte aligned; the accumulator always is
  if ((reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const long long n8 = n >> 3;
    const float4* a4 = reinterpret_cast<const float4*>(acc);
    uint4* o4 = reinterpret_cast<uint4*>(out);
    for (long long k = i; k < n8; k += stride) {
      const float4 lo = __ldcs(a4 + 2 * k), hi = __ldcs(a4 + 2 * k + 1);
      const float f[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      o4[k] = make_uint4(Dt<T>::pack(f), Dt<T>::pack(f + 2), Dt<T>::pack(f + 4),
                         Dt<T>::pack(f + 6));
    }
    i += n8 << 3;
  }
  for (; i < n; i += stride) out[i] = Dt<T>::from_f(acc[i]);
}

// the bwd_stage switch at 0 writes grad_offset / grad_mask directly
static int env_stage() { return options().bwd_stage != 0; }

template <typename T>
static cudaError_t launch_bwd_t(const KParams& kp, int cpt, const void* gout, const void* in,
                                const void* off, const void* msk, float* gin_acc, void* gin,
                                void* goff, void* gmask, cudaStream_t s) {
  const int block = 256;
  const T* go_ = static_cast<const T*>(gout);
  const T* i_ = static_cast<const T*>(in);
  const T* o_ = static_cast<const T*>(off);
  const T* m_ = static_cast<const T*>(msk);
  T* goff_ = static_cast<T*>(goff);
  T* gm_ = static_cast<T*>(gmask);
  const long long items = cpt > 0 ? kp.units * (kp.gc / cpt) : kp.units;
  const long long grid = (items + block - 1) / block;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  switch (cpt) {
#define DCN_CASE(K)                                                                        \
    case K: {                                                                              \
      const size_t st = (size_t)(block / (kp.gc / K)) * kp.P * 3 * sizeof(T);             \
      const int stage = st <= 48 * 1024 && !kp.merged && env_stage();                                    \
      bwd_kernel<T, K><<<(unsigned)grid, block, stage ? st : 0, s>>>(                      \
          kp, go_, i_, o_, m_, gin_acc, goff_, gm_, stage);                                \
      break;                                                                               \
    }
    DCN_CASE(1) DCN_CASE(2) DCN_CASE(4) DCN_CASE(8) DCN_CASE(16) DCN_CASE(32)
#undef DCN_CASE
    case 0:
      bwd_generic_kernel<T><<<(unsigned)grid, block, 0, s>>>(kp, go_, i_, o_, m_, gin_acc, goff_,
                                                             gm_);
      break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((void*)gin_acc != gin) {
    const long long n = (long long)kp.N * kp.H * kp.W * kp.C;
    long long rg = (n + block - 1) / block;
    if (rg > 148LL * 64) rg = 148LL * 64;
    if (rg > 0) round_kernel<T><<<(unsigned)rg, block, 0, s>>>(gin_acc, static_cast<T*>(gin), n);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_round(int dtype, const float* acc, void* out, long long n, cudaStream_t s) {
  const int block = 256;
  long long rg = (n + block - 1) / block;
  if (rg > 148LL * 64) rg = 148LL * 64;
  if (rg <= 0) return cudaSuccess;
  switch (dtype) {
    case DCN_F16:
      round_kernel<__half><<<(unsigned)rg, block, 0, s>>>(acc, static_cast<__half*>(out), n);
      break;
    case DCN_BF16:
      round_kernel<__nv_bfloat16><<<(unsigned)rg, block, 0, s>>>(
          acc, static_cast<__nv_bfloat16*>(out), n);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd(const KParams& kp, int dtype, int cpt, const void* gout, const void* in,
                       const void* off, const void* msk, float* gin_acc, void* gin, void* goff,
                       void* gmask, cudaStream_t s) {
  switch (dtype) {
    case DCN_F32:
      return launch_bwd_t<float>(kp, cpt, gout, in, off, msk, gin_acc, gin, goff, gmask, s);
    case DCN_F16:
      return launch_bwd_t<__half>(kp, cpt, gout, in, off, msk, gin_acc, gin, goff, gmask, s);
    case DCN_BF16:
      return launch_bwd_t<__nv_bfloat16>(kp, cpt, gout, in, off, msk, gin_acc, gin, goff, gmask,
                                         s);
    default: return cudaErrorInvalidValue;
  }
}

DCN_BOUNDS_READER(bwd)

}  // namespace dcn
