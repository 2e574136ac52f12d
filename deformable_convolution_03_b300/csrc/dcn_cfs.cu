// dcn_cfs.cu -- the centre feature scale between the core op and output_proj.
//
// The InternImage-G walkthrough (section 三, item 5) places a sigmoid gate
// after the core: it mixes the core's output with the centre pixel's own
// projected feature x_proj.  One gate per (pixel, group), from a logit per
// (pixel, group), applied to the group's gc channels:
//     s = 1 / (1 + exp(-logit)),   out = core + s * (x_proj - core)
// (= core * (1 - s) + x_proj * s), in float32, rounded once to the storage
// type.  The backward gives
//     d core = g * (1 - s),   d x_proj = g * s,
//     d logit = s * (1 - s) * sum over the group's channels of g * (x_proj - core).
// Both are streaming element-wise passes bound by HBM.  A thread takes a chunk
// of V consecutive channels (16 bytes when the group's channels and the
// pointers allow), so a warp reads whole lines; in the backward the L = gc / V
// lanes of a group sum their partial dot products by shuffles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {
namespace {

template <typename T> __device__ __forceinline__ float cvt_in(T v);
template <> __device__ __forceinline__ float cvt_in<float>(float v) { return v; }
template <> __device__ __forceinline__ float cvt_in<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float cvt_in<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T cvt_out(float v);
template <> __device__ __forceinline__ float cvt_out<float>(float v) { return v; }
template <> __device__ __forceinline__ __half cvt_out<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// V elements moved as one aligned access (16, 8, 4 or 2 bytes)
template <typename T, int V> struct alignas(V * sizeof(T)) Pack {
  T v[V];
};

template <typename T, int V>
__device__ __forceinline__ void load_v(const T* p, float (&f)[V]) {
  const Pack<T, V> k = *reinterpret_cast<const Pack<T, V>*>(p);
#pragma unroll
  for (int i = 0; i < V; ++i) f[i] = cvt_in<T>(k.v[i]);
}
template <typename T, int V>
__device__ __forceinline__ void store_v(T* p, const float (&f)[V]) {
  Pack<T, V> k;
#pragma unroll
  for (int i = 0; i < V; ++i) k.v[i] = cvt_out<T>(f[i]);
  *reinterpret_cast<Pack<T, V>*>(p) = k;
}

__device__ __forceinline__ float gate(float l) { return cfs_gate(l); }

// One thread per chunk of V channels; V divides gc.  out may be core or x_proj
// (each element is read and written by one thread, reads first).
template <typename T, int V>
__global__ void __launch_bounds__(256)
cfs_fwd_kernel(long long chunks, int C, int gc, const T* core, const T* x, const T* logit,
               T* out) {
  const int cpr = C / V;  // chunks per row
  const int G = C / gc;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < chunks;
       k += (long long)gridDim.x * blockDim.x) {
    const long long m = k / cpr;
    const int c = (int)(k - m * cpr) * V;
    const float s = gate(cvt_in<T>(logit[m * G + c / gc]));
    const long long e = m * C + c;
    float a[V], b[V], o[V];
    load_v<T, V>(core + e, a);
    load_v<T, V>(x + e, b);
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = fmaf(s, b[i] - a[i], a[i]);
    store_v<T, V>(out + e, o);
  }
}

// One thread per chunk; the L = gc / V chunks of a (pixel, group) sit in L
// consecutive lanes (L a power of two <= 32; groups start at multiples of L
// chunks and a warp's first chunk is a multiple of 32), whose partial sums
// meet by butterfly shuffles.  The stride loop runs to the chunk count rounded
// up to whole warps, so all lanes of a warp make the same trips and reach the
// shuffles together; lanes past the end take part with zeros.
template <typename T, int V, int L>
__global__ void __launch_bounds__(256)
cfs_bwd_kernel(long long chunks, int C, int gc, const T* gout, const T* core, const T* x,
               const T* logit, T* gcore, T* gx, T* glogit) {
  const int cpr = C / V;
  const int G = C / gc;
  const long long kend = (chunks + 31) / 32 * 32;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < kend;
       k += (long long)gridDim.x * blockDim.x) {
    const bool live = k < chunks;
    float part = 0.f, s = 0.f;
    long long m = 0;
    int c = 0;
    if (live) {
      m = k / cpr;
      c = (int)(k - m * cpr) * V;
      s = gate(cvt_in<T>(logit[m * G + c / gc]));
      const long long e = m * C + c;
      float g[V], a[V], b[V], oc[V], ox[V];
      load_v<T, V>(gout + e, g);
      load_v<T, V>(core + e, a);
      load_v<T, V>(x + e, b);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        part = fmaf(g[i], b[i] - a[i], part);
        oc[i] = g[i] * (1.f - s);
        ox[i] = g[i] * s;
      }
      store_v<T, V>(gcore + e, oc);
      store_v<T, V>(gx + e, ox);
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (live && c % gc == 0) glogit[m * G + c / gc] = cvt_out<T>(s * (1.f - s) * part);
  }
}

// Any gc: one thread per (pixel, group), its channels one by one.
template <typename T>
__global__ void __launch_bounds__(256)
cfs_bwd_group_kernel(long long units, int C, int gc, const T* gout, const T* core, const T* x,
                     const T* logit, T* gcore, T* gx, T* glogit) {
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units;
       u += (long long)gridDim.x * blockDim.x) {
    const float s = gate(cvt_in<T>(logit[u]));
    const long long e0 = u * gc;  // rows are G groups of gc channels, back to back
    float part = 0.f;
    for (int i = 0; i < gc; ++i) {
      const float g = cvt_in<T>(gout[e0 + i]), a = cvt_in<T>(core[e0 + i]);
      const float b = cvt_in<T>(x[e0 + i]);
      part = fmaf(g, b - a, part);
      gcore[e0 + i] = cvt_out<T>(g * (1.f - s));
      gx[e0 + i] = cvt_out<T>(g * s);
    }
    glogit[u] = cvt_out<T>(s * (1.f - s) * part);
  }
}

int grid_for(long long n, int sms) {
  const long long blocks = (n + 255) / 256;
  const long long cap = (long long)sms * 8;
  return (int)(blocks < cap ? blocks : cap);
}

int sm_count() {
  static int n = [] {
    int d = 0, v = 0;
    if (cudaGetDevice(&d) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
      return 148;
    return v;
  }();
  return n;
}

template <typename T, int V>
cudaError_t fwd_v(long long M, int C, int gc, const void* core, const void* x, const void* l,
                  void* out, cudaStream_t st) {
  const long long chunks = M * (C / V);
  cfs_fwd_kernel<T, V><<<grid_for(chunks, sm_count()), 256, 0, st>>>(
      chunks, C, gc, static_cast<const T*>(core), static_cast<const T*>(x),
      static_cast<const T*>(l), static_cast<T*>(out));
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_t(int vbytes, long long M, int C, int gc, const void* core, const void* x,
                  const void* l, void* out, cudaStream_t st) {
  constexpr int es = (int)sizeof(T);
  switch (vbytes / es) {
    case 16 / es: return fwd_v<T, 16 / es>(M, C, gc, core, x, l, out, st);
    case 8 / es: return fwd_v<T, 8 / es>(M, C, gc, core, x, l, out, st);
    case 4 / es: return fwd_v<T, 4 / es>(M, C, gc, core, x, l, out, st);
    default: return fwd_v<T, 1>(M, C, gc, core, x, l, out, st);
  }
}

template <typename T, int V, int L>
cudaError_t bwd_vl(long long M, int C, int gc, const void* go, const void* core, const void* x,
                   const void* l, void* gc_, void* gx, void* gl, cudaStream_t st) {
  const long long chunks = M * (C / V);
  cfs_bwd_kernel<T, V, L><<<grid_for(chunks, sm_count()), 256, 0, st>>>(
      chunks, C, gc, static_cast<const T*>(go), static_cast<const T*>(core),
      static_cast<const T*>(x), static_cast<const T*>(l), static_cast<T*>(gc_),
      static_cast<T*>(gx), static_cast<T*>(gl));
  return cudaGetLastError();
}

template <typename T, int V>
cudaError_t bwd_v(long long M, int C, int gc, const void* go, const void* core, const void* x,
                  const void* l, void* gc_, void* gx, void* gl, cudaStream_t st) {
  switch (gc / V) {
    case 1: return bwd_vl<T, V, 1>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    case 2: return bwd_vl<T, V, 2>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    case 4: return bwd_vl<T, V, 4>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    case 8: return bwd_vl<T, V, 8>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    case 16: return bwd_vl<T, V, 16>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    default: return bwd_vl<T, V, 32>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
  }
}

template <typename T>
cudaError_t bwd_t(int vbytes, long long M, int C, int gc, const void* go, const void* core,
                  const void* x, const void* l, void* gc_, void* gx, void* gl, cudaStream_t st) {
  constexpr int es = (int)sizeof(T);
  if (vbytes > 0) {
    switch (vbytes / es) {
      case 16 / es: return bwd_v<T, 16 / es>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
      case 8 / es: return bwd_v<T, 8 / es>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
      case 4 / es: return bwd_v<T, 4 / es>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
      default: return bwd_v<T, 1>(M, C, gc, go, core, x, l, gc_, gx, gl, st);
    }
  }
  const long long units = M * (C / gc);
  cfs_bwd_group_kernel<T><<<grid_for(units, sm_count()), 256, 0, st>>>(
      units, C, gc, static_cast<const T*>(go), static_cast<const T*>(core),
      static_cast<const T*>(x), static_cast<const T*>(l), static_cast<T*>(gc_),
      static_cast<T*>(gx), static_cast<T*>(gl));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cfs_fwd(int dtype, int vbytes, long long M, int C, int G, const void* core,
                           const void* x, const void* logits, void* out, cudaStream_t st) {
  const int gc = C / G;
  switch (dtype) {
    case DCN_F32: return fwd_t<float>(vbytes, M, C, gc, core, x, logits, out, st);
    case DCN_F16: return fwd_t<__half>(vbytes, M, C, gc, core, x, logits, out, st);
    default: return fwd_t<__nv_bfloat16>(vbytes, M, C, gc, core, x, logits, out, st);
  }
}

cudaError_t launch_cfs_bwd(int dtype, int vbytes, long long M, int C, int G, const void* gout,
                           const void* core, const void* x, const void* logits, void* gcore,
                           void* gx, void* glogits, cudaStream_t st) {
  const int gc = C / G;
  switch (dtype) {
    case DCN_F32:
      return bwd_t<float>(vbytes, M, C, gc, gout, core, x, logits, gcore, gx, glogits, st);
    case DCN_F16:
      return bwd_t<__half>(vbytes, M, C, gc, gout, core, x, logits, gcore, gx, glogits, st);
    default:
      return bwd_t<__nv_bfloat16>(vbytes, M, C, gc, gout, core, x, logits, gcore, gx, glogits,
                                  st);
  }
}

}  // namespace dcn
