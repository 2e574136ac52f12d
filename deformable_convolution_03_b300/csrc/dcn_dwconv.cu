// dcn_dwconv.cu -- the offset branch's feature step in one pass: a k x k
// depthwise convolution (zero padding (k-1)/2, per-channel bias), LayerNorm
// over the channels of each pixel and the exact GELU,
//     x1 = GELU(LayerNorm(dwconv(x))),
// the control features from which the DCN module predicts its offsets and
// mask (page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读",
// section 三 item 2; dw_kernel_size 5 in the page's configuration table).
//
// Tiled kernel (k of 3 or 5, C of 64, 128, 256 or 512).  The image is
// cut into tiles of TH x TW pixels, all C channels; a persistent block takes
// tiles in turn and stages the next tile's input footprint
// (TH+k-1) x (TW+k-1) x C, zeros outside the image, into the other of two
// shared-memory buffers with asynchronous 16-byte copies while it computes the
// current one.  A thread owns a patch of PY x 4 pixels and two channels: it
// holds its channels' k*k weights in registers, walks the footprint rows of
// its patch once and keeps its float32 sums as channel pairs, updated with
// packed two-lane FMAs.  The C / 2 threads of a patch then reduce the
// LayerNorm statistics of its pixels: a butterfly over the warp's 32 lanes
// leaves each pixel's sum on 32 / (4 PY) lanes, the patch's warps add their
// sums through shared memory, and the mean and later the inverse deviation
// are broadcast back by shuffles.  The mean comes first and the variance is
// then summed over the deviations held in registers (two passes, no
// cancellation).  Each thread normalises, applies gamma, beta and the GELU
// (erf by a published rational approximation, below) and stores its two
// channels of each pixel once, rounded to the
// storage type.  The input is read from memory once (halos come from L2) and
// the output written once.
//
// General kernel (any odd k, any C up to 2048): one warp per pixel, lanes over
// channels, the k*k taps read through L1, the pixel's C sums kept in shared
// memory between the passes.
#include <climits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {
namespace {

constexpr int kPX = 4;  // a patch is PY x kPX pixels

// Two consecutive elements of T as float32.
template <typename T> __device__ __forceinline__ float2 two_f(const T* p);
template <> __device__ __forceinline__ float2 two_f<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <> __device__ __forceinline__ float2 two_f<__half>(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}
template <> __device__ __forceinline__ float2 two_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <typename T> __device__ __forceinline__ void put_two(T* p, float2 v);
template <> __device__ __forceinline__ void put_two<float>(float* p, float2 v) {
  *reinterpret_cast<float2*>(p) = v;
}
template <> __device__ __forceinline__ void put_two<__half>(__half* p, float2 v) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}
template <> __device__ __forceinline__ void put_two<__nv_bfloat16>(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// The hardware's approximate reciprocal and base-2 exponential (relative
// error a few 2^-23; results below 2^-126 flush to zero).
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// GELU, z * Phi(z), with erf from Abramowitz and Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (|error| <= 1.5e-7 for all
// arguments): for u >= 0, erf(u) = 1 - q(u) with
//     q(u) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-u^2),
//     t = 1 / (1 + p u).
// With u = |z| / sqrt(2), z Phi(z) = z (1 + sign(z) erf(u)) / 2 becomes
//     GELU(z) = max(z, 0) - |z| q(u) / 2
// for either sign, without branches.  The error in GELU is at most
// |z| * 0.75e-7 plus float32 rounding; where exp(-u^2) falls below 2^-126
// (|z| > 13) the term is dropped, an error below 1e-36.
constexpr float kAsP = 0.3275911f * 0.70710678118654752f;  // p / sqrt(2): t from |z|
constexpr float kAsE = -0.72134752044448170f;               // -log2(e) / 2: 2^(kAsE z^2) = exp(-u^2)
constexpr float kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                kA4 = -1.453152027f, kA5 = 1.061405429f;

// GELU of two values (packed float32 pairs where the arithmetic allows).
__device__ __forceinline__ float2 gelu2(float2 z) {
  const float2 t = make_float2(rcp_approx(fmaf(kAsP, fabsf(z.x), 1.f)),
                               rcp_approx(fmaf(kAsP, fabsf(z.y), 1.f)));
  float2 q = __ffma2_rn(t, make_float2(kA5, kA5), make_float2(kA4, kA4));
  q = __ffma2_rn(t, q, make_float2(kA3, kA3));
  q = __ffma2_rn(t, q, make_float2(kA2, kA2));
  q = __ffma2_rn(t, q, make_float2(kA1, kA1));
  const float2 a = __fmul2_rn(__fmul2_rn(z, make_float2(kAsE, kAsE)), z);
  q = __fmul2_rn(__fmul2_rn(t, q), make_float2(ex2_approx(a.x), ex2_approx(a.y)));
  return make_float2(fmaf(-0.5f * fabsf(z.x), q.x, fmaxf(z.x, 0.f)),
                     fmaf(-0.5f * fabsf(z.y), q.y, fmaxf(z.y, 0.f)));
}

// The same GELU for one value.
__device__ __forceinline__ float gelu1(float z) {
  const float t = rcp_approx(fmaf(kAsP, fabsf(z), 1.f));
  float q = fmaf(t, kA5, kA4);
  q = fmaf(t, q, kA3);
  q = fmaf(t, q, kA2);
  q = fmaf(t, q, kA1);
  q = t * q * ex2_approx(kAsE * z * z);
  return fmaf(-0.5f * fabsf(z), q, fmaxf(z, 0.f));
}

// 16 bytes from global to shared memory, asynchronously; bytes = 0 fills the
// 16 bytes with zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Butterfly sum of v[0..NP) over the warp's 32 lanes (NP of 8 or 16): each
// step trades half of the values with the lane o apart, so that after
// log2(NP) steps lane l holds pixel (l / (32 / NP)) % NP summed over the
// lanes that differ in those bits; the remaining bits are summed plainly.
// Returns that pixel's warp total (on all 32 / NP lanes that hold it).
template <int NP>
__device__ __forceinline__ float warp_sum(float (&v)[NP], int lane) {
#pragma unroll
  for (int half = NP / 2, o = 16; half >= 1; half >>= 1, o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i];
      const float send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float s = v[0];
#pragma unroll
  for (int o = 16 / NP; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// The patch's total of a per-pixel quantity: the warp sums, then (nw > 1) the
// sums of the patch's nw warps through red[patch][NP][nw].  Every thread of
// the block calls it (it may synchronise the block).
template <int NP>
__device__ __forceinline__ float patch_sum(float (&v)[NP], int lane, int wi, int nw, int patch,
                                           float* red) {
  const float s = warp_sum<NP>(v, lane);
  if (nw == 1) return s;
  constexpr int LS = 32 / NP;
  const int p = (lane / LS) % NP;
  float* r = red + ((size_t)patch * NP + p) * nw;
  if (lane % LS == 0) r[wi] = s;
  __syncthreads();
  float t = 0.f;
  for (int q = 0; q < nw; ++q) t += r[q];
  return t;
}

template <typename T, int K, int PY, int C>
__global__ void __launch_bounds__(256, 2)
dwconv_tile_kernel(const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ bias,
                   const T* __restrict__ gamma, const T* __restrict__ beta, T* __restrict__ y,
                   int H, int W, float eps, int pw, int tiles_w, int tiles, int total) {
  constexpr int R = (K - 1) / 2;
  constexpr int NP = PY * kPX;             // pixels of a patch
  constexpr int IW = kPX + K - 1;          // footprint columns of a patch
  constexpr int kV = 16 / (int)sizeof(T);  // elements of a 16-byte copy
  constexpr int S = C / 2;                 // threads of a patch (two channels each)
  constexpr int NW = S / 32;               // warps of a patch
  constexpr int CV = C / kV;               // 16-byte copies per pixel
  extern __shared__ __align__(16) unsigned char smem[];
  const int npatch = blockDim.x / S;  // patches of the block
  const int th = (npatch / pw) * PY, tw = pw * kPX;
  const int fh = th + K - 1, fw = tw + K - 1;
  const int foot_bytes = (fh * fw * C * (int)sizeof(T) + 15) / 16 * 16;
  float* red = reinterpret_cast<float*>(smem + 2 * foot_bytes);
  float* red2 = red + npatch * NP * NW;
  const uint32_t smem_base = (uint32_t)__cvta_generic_to_shared(smem);

  // this thread's 16-byte slot within a pixel of the footprint, and the
  // pixels it copies: tid / CV, then every ppi further
  const int ppi = blockDim.x / CV;
  const int vec = threadIdx.x % CV, pix0 = threadIdx.x / CV;
  const int nfoot = fh * fw;
  const int fi0 = pix0 / fw, fj0 = pix0 - fi0 * fw;  // first pixel copied
  const int dfi = ppi / fw, dfj = ppi - dfi * fw;    // the step between pixels copied
  const size_t x_bytes = (size_t)(total / tiles) * H * W * C * sizeof(T);  // (checked build)
  auto stage = [&](int t, int buf) {
    const int n = t / tiles;
    const int tile = t - n * tiles;
    const int ty = tile / tiles_w;
    const int i0 = ty * th - R, j0 = (tile - ty * tiles_w) * tw - R;
    const T* xn = x + (size_t)n * H * W * C + vec * kV;
    uint32_t dst = smem_base + (uint32_t)(buf * foot_bytes) + (uint32_t)(pix0 * C + vec * kV) * sizeof(T);
    const uint32_t dstep = (uint32_t)(ppi * C * sizeof(T));
    int i = i0 + fi0, j = j0 + fj0;
    for (int pix = pix0; pix < nfoot; pix += ppi, dst += dstep) {
      bool in = (unsigned)i < (unsigned)H && (unsigned)j < (unsigned)W;
      const T* src = xn + ((size_t)i * W + j) * C;
      if (in && !DCN_IN_SPAN(src, 16, x, x_bytes, kBadStage)) in = false;
      if (DCN_IN_SPAN(reinterpret_cast<const void*>((uintptr_t)dst), 16,
                      reinterpret_cast<const void*>((uintptr_t)(smem_base + buf * foot_bytes)),
                      foot_bytes, kBadStage))
        cp_async16(dst, in ? (const void*)src : (const void*)x, in ? 16u : 0u);
      i += dfi;
      j += dfj;
      if (j >= j0 + fw) {
        j -= fw;
        ++i;
      }
    }
    cp_async_commit();
  };

  const int s = threadIdx.x % S, patch = threadIdx.x / S;
  const int lane = threadIdx.x & 31, wi = s >> 5;
  const int c0 = 2 * s;
  const int pi = (patch / pw) * PY, pj = (patch % pw) * kPX;  // patch origin in the tile

  int t = blockIdx.x;
  if (t < total) stage(t, 0);
  float2 wt[K][K];
#pragma unroll
  for (int a = 0; a < K; ++a)
#pragma unroll
    for (int e = 0; e < K; ++e) wt[a][e] = two_f<T>(w + (a * K + e) * C + c0);
  const float2 b0 = bias ? two_f<T>(bias + c0) : make_float2(0.f, 0.f);
  const float2 g = two_f<T>(gamma + c0), bt = two_f<T>(beta + c0);
  constexpr float kInvC = 1.f / (float)C;

  for (int it = 0; t < total; ++it, t += gridDim.x) {
    const int buf = it & 1;
    if (t + (int)gridDim.x < total) {
      stage(t + gridDim.x, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const T* foot = reinterpret_cast<const T*>(smem + buf * foot_bytes) + (pi * fw + pj) * C + c0;

    float2 acc[PY][kPX];
#pragma unroll
    for (int py = 0; py < PY; ++py)
#pragma unroll
      for (int px = 0; px < kPX; ++px) acc[py][px] = b0;
    // footprint row fr feeds output row py through kernel row a = fr - py
#pragma unroll
    for (int fr = 0; fr < PY + K - 1; ++fr) {
      const T* row = foot + fr * fw * C;
      float2 in[IW];
#pragma unroll
      for (int q = 0; q < IW; ++q)
        in[q] = DCN_IN_SPAN(row + q * C, 2 * sizeof(T), smem + buf * foot_bytes, foot_bytes,
                            kBadShared)
                    ? two_f<T>(row + q * C)
                    : make_float2(0.f, 0.f);
#pragma unroll
      for (int py = 0; py < PY; ++py) {
        const int a = fr - py;
        if (a < 0 || a >= K) continue;
#pragma unroll
        for (int e = 0; e < K; ++e)
#pragma unroll
          for (int px = 0; px < kPX; ++px) acc[py][px] = __ffma2_rn(wt[a][e], in[px + e], acc[py][px]);
      }
    }

    // LayerNorm statistics of the patch's pixels: the mean, then the mean
    // square deviation, both over the C channels
    float v[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) v[q] = acc[q / kPX][q % kPX].x + acc[q / kPX][q % kPX].y;
    const float mean_p = patch_sum<NP>(v, lane, wi, NW, patch, red) * kInvC;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const float m = -__shfl_sync(0xffffffffu, mean_p, q * (32 / NP));
      const float2 d = __fadd2_rn(acc[q / kPX][q % kPX], make_float2(m, m));
      acc[q / kPX][q % kPX] = d;
      v[q] = fmaf(d.x, d.x, d.y * d.y);
    }
    const float var_p = patch_sum<NP>(v, lane, wi, NW, patch, red2) * kInvC;
    const float inv_p = 1.f / sqrtf(var_p + eps);

#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const float inv = __shfl_sync(0xffffffffu, inv_p, q * (32 / NP));
      const float2 z = __ffma2_rn(__fmul2_rn(acc[q / kPX][q % kPX], make_float2(inv, inv)), g, bt);
      acc[q / kPX][q % kPX] = gelu2(z);
    }
    const int n = t / tiles;
    const int tile = t - n * tiles;
    const int ty = tile / tiles_w;
    const int i0 = ty * th + pi, j0 = (tile - ty * tiles_w) * tw + pj;
    T* yp = y + (((size_t)n * H + i0) * W + j0) * C + c0;
    const size_t row = (size_t)W * C;
    if (i0 + PY <= H && j0 + kPX <= W) {
#pragma unroll
      for (int py = 0; py < PY; ++py, yp += row)
#pragma unroll
        for (int px = 0; px < kPX; ++px)
          if (DCN_IN_SPAN(yp + px * C, 2 * sizeof(T), y, x_bytes, kBadStore))
            put_two<T>(yp + px * C, acc[py][px]);
    } else {
#pragma unroll
      for (int py = 0; py < PY; ++py, yp += row)
#pragma unroll
        for (int px = 0; px < kPX; ++px)
          if (i0 + py < H && j0 + px < W &&
              DCN_IN_SPAN(yp + px * C, 2 * sizeof(T), y, x_bytes, kBadStore))
            put_two<T>(yp + px * C, acc[py][px]);
    }
    __syncthreads();  // this buffer and red are rewritten in the next turn
  }
}

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_f<__half>(const __half* p) {
  return __half2float(__ldg(p));
}
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}
template <typename T> __device__ __forceinline__ T st_f(float v);
template <> __device__ __forceinline__ float st_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half st_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 st_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// One warp per pixel; the pixel's C float32 sums sit in the warp's C floats of
// shared memory between the passes.
constexpr int kGenWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kGenWarps * 32)
dwconv_general_kernel(const T* __restrict__ x, const T* __restrict__ w,
                      const T* __restrict__ bias, const T* __restrict__ gamma,
                      const T* __restrict__ beta, T* __restrict__ y, long long pixels, int H,
                      int W, int C, int k, float eps) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  float* buf = reinterpret_cast<float*>(smem) + (size_t)wi * C;
  const long long m = (long long)blockIdx.x * kGenWarps + wi;
  if (m >= pixels) return;  // the whole warp leaves; no block barrier follows
  const int r = (k - 1) / 2;
  const long long nhw = m / W;
  const int j = (int)(m - nhw * W);
  const int i = (int)(nhw % H);
  const long long n = nhw / H;
  const T* xn = x + (size_t)n * H * W * C;
  float s = 0.f;
  for (int c = lane; c < C; c += 32) {
    float acc = bias ? ld_f<T>(bias + c) : 0.f;
    for (int a = 0; a < k; ++a) {
      const int ii = i + a - r;
      if ((unsigned)ii >= (unsigned)H) continue;
      for (int e = 0; e < k; ++e) {
        const int jj = j + e - r;
        if ((unsigned)jj >= (unsigned)W) continue;
        const T* src = xn + ((size_t)ii * W + jj) * C + c;
        if (!DCN_IN_SPAN(src, sizeof(T), x, (size_t)pixels * C * sizeof(T), kBadGather)) continue;
        acc = fmaf(ld_f<T>(w + (size_t)(a * k + e) * C + c), ld_f<T>(src), acc);
      }
    }
    buf[c] = acc;
    s += acc;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / (float)C;
  float s2 = 0.f;
  for (int c = lane; c < C; c += 32) {
    const float d = buf[c] - mean;
    s2 = fmaf(d, d, s2);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  const float inv = 1.f / sqrtf(s2 / (float)C + eps);
  T* ym = y + (size_t)m * C;
  if (!DCN_IN_SPAN(ym, C * sizeof(T), y, (size_t)pixels * C * sizeof(T), kBadStore)) return;
  for (int c = lane; c < C; c += 32) {
    const float z = fmaf((buf[c] - mean) * inv, ld_f<T>(gamma + c), ld_f<T>(beta + c));
    ym[c] = st_f<T>(gelu1(z));
  }
}

template <typename T, int K, int PY, int C>
cudaError_t launch_tiled(const DwGeom& d, const T* x, const T* w, const T* b, const T* g,
                         const T* bt, T* y, cudaStream_t st) {
  const int th = d.ph * PY, tw = d.pw * kPX;
  const int tiles_w = (d.W + tw - 1) / tw, tiles_h = (d.H + th - 1) / th;
  const long long total = (long long)d.N * tiles_w * tiles_h;
  if (total > INT_MAX / 2) return cudaErrorInvalidConfiguration;
  const size_t smem = dwconv_smem_bytes(d, (int)sizeof(T));
  auto kern = dwconv_tile_kernel<T, K, PY, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int threads = d.ph * d.pw * (C / 2);
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem)) !=
      cudaSuccess)
    return e;
  const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(total < cap ? total : cap);
  kern<<<grid, threads, smem, st>>>(x, w, b, g, bt, y, d.H, d.W, d.eps, d.pw, tiles_w,
                                    tiles_w * tiles_h, (int)total);
  return cudaGetLastError();
}

template <typename T, int K, int PY>
cudaError_t launch_tiled_c(const DwGeom& d, const T* x, const T* w, const T* b, const T* g,
                           const T* bt, T* y, cudaStream_t st) {
  switch (d.C) {
    case 64: return launch_tiled<T, K, PY, 64>(d, x, w, b, g, bt, y, st);
    case 128: return launch_tiled<T, K, PY, 128>(d, x, w, b, g, bt, y, st);
    case 256: return launch_tiled<T, K, PY, 256>(d, x, w, b, g, bt, y, st);
    case 512: return launch_tiled<T, K, PY, 512>(d, x, w, b, g, bt, y, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_t(const DwGeom& d, const void* x, const void* w, const void* b, const void* g,
                     const void* bt, void* y, cudaStream_t st) {
  const T* x_ = static_cast<const T*>(x);
  const T* w_ = static_cast<const T*>(w);
  const T* b_ = static_cast<const T*>(b);
  const T* g_ = static_cast<const T*>(g);
  const T* bt_ = static_cast<const T*>(bt);
  T* y_ = static_cast<T*>(y);
  if (d.tiled) {
    if (d.k == 3)
      return d.py == 4 ? launch_tiled_c<T, 3, 4>(d, x_, w_, b_, g_, bt_, y_, st)
                       : launch_tiled_c<T, 3, 2>(d, x_, w_, b_, g_, bt_, y_, st);
    return d.py == 4 ? launch_tiled_c<T, 5, 4>(d, x_, w_, b_, g_, bt_, y_, st)
                     : launch_tiled_c<T, 5, 2>(d, x_, w_, b_, g_, bt_, y_, st);
  }
  const long long pixels = (long long)d.N * d.H * d.W;
  const long long grid = (pixels + kGenWarps - 1) / kGenWarps;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  const size_t smem = dwconv_smem_bytes(d, (int)sizeof(T));
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        dwconv_general_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dwconv_general_kernel<T><<<(unsigned)grid, kGenWarps * 32, smem, st>>>(
      x_, w_, b_, g_, bt_, y_, pixels, d.H, d.W, d.C, d.k, d.eps);
  return cudaGetLastError();
}

}  // namespace

DCN_BOUNDS_READER(dwconv)

size_t dwconv_smem_bytes(const DwGeom& d, int es) {
  if (!d.tiled) return (size_t)kGenWarps * d.C * sizeof(float);
  const size_t fh = (size_t)d.ph * d.py + d.k - 1, fw = (size_t)d.pw * kPX + d.k - 1;
  const size_t foot = (fh * fw * d.C * es + 15) / 16 * 16;
  return 2 * foot + 2 * (size_t)d.ph * d.pw * (d.py * kPX) * (d.C / 64) * sizeof(float);
}

cudaError_t launch_dwconv(const DwGeom& d, int dtype, const void* x, const void* w, const void* b,
                          const void* g, const void* bt, void* y, cudaStream_t s) {
  switch (dtype) {
    case DCN_F32: return launch_t<float>(d, x, w, b, g, bt, y, s);
    case DCN_F16: return launch_t<__half>(d, x, w, b, g, bt, y, s);
    case DCN_BF16: return launch_t<__nv_bfloat16>(d, x, w, b, g, bt, y, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dcn
