// dcn_common.cuh -- internal definitions shared by the forward and backward
// kernels of libdcn_b300: the kernel parameter record, storage-dtype traits and
// vector loads / stores of a thread's channel slice.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/dcn_core.h"

namespace dcn {

// Unsigned division by a runtime-invariant divisor d as a multiply and a shift
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up variant): with s = ceil(log2 d) and
// mul = floor(2^32 (2^s - d) / d) + 1, n / d = (umulhi(n, mul) + n) >> s for
// every n < 2^31 (the sum stays below 2^32).
struct FastDiv {
  uint32_t mul, shift, d;
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return (__umulhi(n, mul) + n) >> shift;
  }
};

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
  FastDiv div_G, div_Wo, div_Ho;
  // 2-D tiling of the wide forward: a block covers tile_w x tile_h output
  // pixels (all groups and channel slices of each); 0 means linear order.
  int tile_w, tile_h, tiles_w, tiles_h;
  // Elements between consecutive units' offset rows and mask rows: 2P and P
  // for separate tensors; the row stride of the merged offset/mask tensor
  // (mask = offset + 2P) when merged != 0, whose gradient rows then also get
  // their padding (elements 3P .. stride-1) written as zero.
  int os_off, os_mask, merged;
  // merged rows that start 32-byte aligned, 16-bit storage, P = 9: the wide
  // forward reads the first 64 bytes of a row (2P offsets, then P masks) with
  // two 256-bit loads instead of one load per value
  int merged_rows64;
  // Kernel taps of the P points, in point order (x-major, centre removed when
  // asked): ix*dilation_w - cen_w and iy*dilation_h - cen_h, as floats (exact).
  float tap_x[DCN_MAX_POINTS];
  float tap_y[DCN_MAX_POINTS];
};

// Geometry of the split backward's input blocks (dcn_bwd_split.cu): a CTA owns TH
// x TW output pixels of one (image, group) and a window of WH x WW input
// pixels whose origin, for the tile starting at output (ho0, wo0), is
// (ho0*stride_h + org_y, wo0*stride_w + org_x).
struct WinGeom {
  int TH, TW;
  int tiles_h, tiles_w;
  int WH, WW;
  int org_y, org_x;
  // 1 when one tile covers each (image, group) plane and its window covers
  // every bilinear cell that touches the image: the plane's grad_input then
  // comes from one block alone, which writes it in the storage type directly
  // (no float32 accumulator to clear, reduce into and round)
  int direct;
};

// Geometry of the TMA-staged forward (fwd_tile_kernel): a block covers the
// output tile of kp (tile_w x tile_h pixels) for GB consecutive groups, and
// loads the input window of WH x WW pixels x GB*gc channels at
// (ho0*stride_h + org_y, wo0*stride_w + org_x) into shared memory with one
// tensor copy; ngb = G / GB blocks cover the groups of a tile.
struct TileGeom {
  int GB, ngb;
  int WH, WW;
  int org_y, org_x;
  unsigned win_bytes;
};

// The forward with its offset/mask projection (dcn_fwd_proj.cu): K = 64 * KB
// feature channels, row_stride rs, NB = GB * rs projection outputs per block
// (tensor-memory columns ncols), the rows in shared memory om_stride elements
// apart; byte offsets of the weight tiles, the window and the barriers in the
// block's shared memory (after 1024-byte alignment), and its total.
struct ProjGeom {
  int KB, rs, NB, ncols, om_stride;
  unsigned b_off, win_off, bar_off, om_bytes, smem_bytes;
  // the persistent, warp-specialised kernel (ws != 0): S feature stages, two
  // windows and two row buffers, their byte offsets and strides; the
  // sampling warps of a block
  int ws, S, sample_warps;
  unsigned a_off, win_stride, rows_off, rows_stride;
};

// Shared memory of bwd_input_kernel: per sample (TH*TW*P), in cell order, its
// four corner weights (4 x 16 bits for 16-bit storage, 4 x float32 otherwise)
// and its 16-bit unit, the tile's grad_out (gc*es bytes per output
// pixel), per-cell counts and list heads ((WH-1)*(WW-1) cells), and 32
// per-warp sums for the scan.
__host__ __device__ inline size_t split_smem_bytes(const WinGeom& wg, int P, int gc, int es) {
  const size_t nunit = (size_t)wg.TH * wg.TW, nsamp = nunit * P;
  const size_t ncell = (size_t)(wg.WH - 1) * (wg.WW - 1);
  auto up16 = [](size_t b) { return (b + 15) / 16 * 16; };
  return up16(nsamp * (es == 2 ? 8 : 16)) + up16(nsamp * 2) + nunit * gc * es +
         (2 * ncell + 1 + 32) * sizeof(int);
}

// The centre feature scale's gate s = 1 / (1 + e^-l) in float32 (its
// forward kernel and the core forward that applies it in its epilogue).
__device__ __forceinline__ float cfs_gate(float l) { return 1.f / (1.f + expf(-l)); }

// ---- asynchronous tensor copies (TMA) and their barrier --------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// one arrival that also announces the bytes the copy will deliver
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of the barrier at most `limit` polls (each poll
// itself blocks for a hardware-defined time); false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int limit) {
  for (int i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// A 4-D tiled copy global -> shared, completing on the barrier; coordinates
// innermost first, out-of-range elements read as zero.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ---- tensor cores (tcgen05) ---------------------------------------------------

// Shared-memory matrix descriptor of tcgen05.mma for a K-major operand in the
// 128-byte swizzled layout: rows of 128 bytes (64 16-bit elements), groups of
// 8 rows 1024 bytes apart.  Fields: start address >> 4 (bits 0-13), leading
// byte offset (unused for this layout, 1), stride byte offset >> 4 (bits
// 32-45), descriptor version 1 (bits 46-47), layout 2 = 128-byte swizzle
// (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: float32 accumulator (bits
// 4-5 = 1), A and B of format fmt (0 = f16, 1 = bf16; bits 7-9 and 10-12),
// both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t fmt, uint32_t n, uint32_t m) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}

// 16 columns of one tensor-memory lane per thread, without waiting: the
// caller issues several, then one tcgen05.wait::ld
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 16 columns at each of two tensor-memory addresses, then the wait, in one
// statement (the registers are defined only after the wait)
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16],
                                            uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, "
      "%25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]),
        "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]),
        "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]),
        "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- range checks (the DCN_DEBUG_BOUNDS build) -------------------------------
// Built with -DDCN_DEBUG_BOUNDS, every data-dependent access (a bilinear
// corner gathered from the input or from a staged window, a grad_input
// scatter, a row read or written at a computed index) first checks that its
// bytes lie inside the tensor or buffer it belongs to.  An access that does
// not is skipped (a load reads zeros) and sets a bit of this translation
// unit's status word; the C ABI layer then synchronises after each call and
// returns DCN_ERR_INTERNAL if any word is non-zero.  Nothing traps.  In the
// normal build the checks compile to nothing and their arguments are dead.

enum : unsigned {
  kBadGather = 1u,   // a corner read from the input tensor
  kBadShared = 2u,   // a read from a staged window or tile in shared memory
  kBadScatter = 4u,  // a grad_input (accumulator) reduction
  kBadStore = 8u,    // an output, grad_offset or grad_mask row
  kBadRow = 16u,     // an offset, mask or upstream-gradient row
  kBadStage = 32u,   // a staging copy's source or destination
};

#ifdef DCN_DEBUG_BOUNDS
namespace {
__device__ unsigned int g_bounds_status;
}
__device__ __forceinline__ bool in_span(const void* p, size_t n, const void* lo, size_t bytes,
                                        unsigned bit) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(lo);
  const bool ok = a >= b && a + n <= b + bytes;
  if (!ok) atomicOr(&g_bounds_status, bit);
  return ok;
}
#define DCN_IN_SPAN(p, n, lo, bytes, bit) ::dcn::in_span((p), (n), (lo), (bytes), (bit))
// This translation unit's reader: copies the status word out and clears it.
#define DCN_BOUNDS_READER(name)                                                          \
  cudaError_t bounds_status_##name(unsigned* v) {                                        \
    const unsigned zero = 0;                                                             \
    cudaError_t e = cudaMemcpyFromSymbol(v, g_bounds_status, sizeof(unsigned));          \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bounds_status, &zero, sizeof zero);   \
    return e;                                                                            \
  }                                                                                      \
  cudaError_t bounds_status_set_##name(unsigned v) {                                     \
    return cudaMemcpyToSymbol(g_bounds_status, &v, sizeof v);                            \
  }
#else
#define DCN_IN_SPAN(p, n, lo, bytes, bit) true
#define DCN_BOUNDS_READER(name)                                                          \
  cudaError_t bounds_status_##name(unsigned* v) {                                        \
    *v = 0;                                                                              \
    return cudaSuccess;                                                                  \
  }                                                                                      \
  cudaError_t bounds_status_set_##name(unsigned) { return cudaSuccess; }
#endif

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
  __device__ __forceinline__ static float to_f(__half v) { return __half2float(v); }
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
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// Loads of data read once (offsets, masks): not kept in L1, so that they do
// not evict the input lines that neighbouring samples reuse.
template <typename T> __device__ __forceinline__ float ld_once_1(const T* p);
template <typename T> __device__ __forceinline__ float2 ld_once_2(const T* p);

template <> __device__ __forceinline__ float ld_once_1<float>(const float* p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
template <> __device__ __forceinline__ float2 ld_once_2<float>(const float* p) {
  float2 v;
  asm("ld.global.nc.L1::no_allocate.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
template <> __device__ __forceinline__ float ld_once_1<__half>(const __half* p) {
  unsigned short h;
  asm("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(h) : "l"(p));
  return __half2float(__ushort_as_half(h));
}
template <> __device__ __forceinline__ float2 ld_once_2<__half>(const __half* p) {
  uint32_t w;
  asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(w) : "l"(p));
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}
template <> __device__ __forceinline__ float ld_once_1<__nv_bfloat16>(const __nv_bfloat16* p) {
  unsigned short h;
  asm("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(h) : "l"(p));
  return __uint_as_float((uint32_t)h << 16);
}
template <> __device__ __forceinline__ float2 ld_once_2<__nv_bfloat16>(const __nv_bfloat16* p) {
  uint32_t w;
  asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(w) : "l"(p));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

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

// A slice gathered from the tensor [lo, lo + bytes) (checked in the
// DCN_DEBUG_BOUNDS build; zeros if it lies outside).
template <typename T, int CPT>
__device__ __forceinline__ void load_slice_in(const T* p, float (&v)[CPT], const void* lo,
                                              size_t bytes) {
  if (!DCN_IN_SPAN(p, CPT * sizeof(T), lo, bytes, kBadGather)) {
#pragma unroll
    for (int i = 0; i < CPT; ++i) v[i] = 0.f;
    return;
  }
  Slice<T, CPT>::load(p, v);
}

// Bytes of the input tensor, and the spans of the offset and mask rows of
// all units (row u starts at u * os elements; the last row ends its 2P or P
// values in; a merged offset/mask tensor holds whole rows of os_off).
template <typename T> __device__ __forceinline__ size_t input_bytes(const KParams& kp) {
  return (size_t)kp.N * kp.H * kp.W * kp.C * sizeof(T);
}
template <typename T> __device__ __forceinline__ size_t offset_bytes(const KParams& kp) {
  return (kp.merged ? (size_t)kp.units * kp.os_off
                    : (size_t)(kp.units - 1) * kp.os_off + 2 * kp.P) * sizeof(T);
}
template <typename T> __device__ __forceinline__ size_t mask_bytes(const KParams& kp) {
  return ((size_t)(kp.units - 1) * kp.os_mask + kp.P) * sizeof(T);
}
// The unit's offset and mask rows lie inside their tensors (always true in
// the normal build).
template <typename T>
__device__ __forceinline__ bool rows_in(const KParams& kp, const T* offset, const T* mask,
                                        const T* orow, const T* mrow) {
  return DCN_IN_SPAN(orow, 2 * kp.P * sizeof(T), offset, offset_bytes<T>(kp), kBadRow) &&
         DCN_IN_SPAN(mrow, kp.P * sizeof(T), mask, mask_bytes<T>(kp), kBadRow);
}
// The unit's row of gc values at out + unit * gc lies inside the output
// (N*Ho*Wo*G rows).
template <typename T>
__device__ __forceinline__ bool out_in(const KParams& kp, const T* out, const T* row, int n) {
  return DCN_IN_SPAN(row, n * sizeof(T), out, (size_t)kp.units * kp.gc * sizeof(T), kBadStore);
}

// ---- wide gathers: NW 32-bit words from a 32-byte-aligned address -----------

template <int NW>
__device__ __forceinline__ void ldg_words(const void* p, uint32_t (&w)[NW]) {
  static_assert(NW % 4 == 0, "16-byte multiples only");
  const char* c = static_cast<const char*>(p);
  if constexpr (NW % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 8; ++i)
      asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
          : "=r"(w[8 * i + 0]), "=r"(w[8 * i + 1]), "=r"(w[8 * i + 2]), "=r"(w[8 * i + 3]),
            "=r"(w[8 * i + 4]), "=r"(w[8 * i + 5]), "=r"(w[8 * i + 6]), "=r"(w[8 * i + 7])
          : "l"(c + 32 * i));
  } else {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      uint4 u = __ldg(reinterpret_cast<const uint4*>(c) + i);
      w[4 * i + 0] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
    }
  }
}

// ldg_words of a corner inside the tensor [lo, lo + bytes) (checked in the
// DCN_DEBUG_BOUNDS build; zeros if it is not).
template <int NW>
__device__ __forceinline__ void ldg_words_in(const void* p, uint32_t (&w)[NW], const void* lo,
                                             size_t bytes) {
  if (!DCN_IN_SPAN(p, 4 * NW, lo, bytes, kBadGather)) {
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = 0u;
    return;
  }
  ldg_words<NW>(p, w);
}

// N consecutive 32-bit words starting at the 4-byte aligned address p, read
// with NV 16-byte loads of the aligned window around them (not kept in L1)
// and shifted into place in registers.  The caller guarantees that the window
// [p & ~15, (p & ~15) + 16*NV) lies inside the tensor; 16*NV >= 4*N + 12.
template <int NV, int N>
__device__ __forceinline__ void words_from_window(const void* p, uint32_t (&out)[N]) {
  static_assert(16 * NV >= 4 * N + 12, "window too small");
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const char* base = reinterpret_cast<const char*>(a & ~uintptr_t(15));
  const int sh = (int)(a & 15) >> 2;  // words to skip, 0..3
  uint32_t w[4 * NV];
#pragma unroll
  for (int i = 0; i < NV; ++i)
    asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
        : "l"(base + 16 * i));
#pragma unroll
  for (int j = 0; j + 2 < 4 * NV; ++j) w[j] = (sh & 2) ? w[j + 2] : w[j];
#pragma unroll
  for (int j = 0; j < N; ++j) out[j] = (sh & 1) ? w[j + 1] : w[j];
}

// The offset row (2P values) and mask row (P values) of one unit in separate
// tensors, for P = KP fixed at compile time, read with a few 16-byte loads of
// the aligned windows around them (words_from_window) instead of one scalar
// load per value.  A warp's lanes hold units whose rows are 2P*es bytes or
// more apart, so each scalar load instruction would touch up to 32 lines.
// load() declines (returns false) when a window would leave its tensor (the
// first or last units of a tensor that is not 16-byte aligned at both ends);
// the caller then reads the values one by one.
template <typename T, int KP>
struct UnitRows {
  static constexpr int kEs = (int)sizeof(T);
  static constexpr int kP = KP > 0 ? KP : 1;
  // offsets: KP words of (dx, dy) 16-bit pairs, or 2*KP float32 words
  static constexpr int NO = kEs == 2 ? kP : 2 * kP;
  static constexpr int NVO = (4 * NO + 12 + 15) / 16;
  // mask: 16-bit values two to a word (value p in half p after the shift),
  // or one float32 per word
  static constexpr int NM = kEs == 2 ? (kP + 2) / 2 : kP;
  static constexpr int NVM = (4 * NM + 12 + 15) / 16;
  uint32_t ow[NO], mw[NM];

  __device__ __forceinline__ bool load(const T* offset, const T* mask, long long units,
                                       const T* orow, const T* mrow) {
    const uintptr_t ob = reinterpret_cast<uintptr_t>(offset);
    const uintptr_t mb = reinterpret_cast<uintptr_t>(mask);
    const uintptr_t oe = ob + (uintptr_t)units * 2 * kP * kEs;
    const uintptr_t me = mb + (uintptr_t)units * kP * kEs;
    const uintptr_t oa = reinterpret_cast<uintptr_t>(orow) & ~uintptr_t(15);
    const uintptr_t mw4 = reinterpret_cast<uintptr_t>(mrow) & ~uintptr_t(3);
    const uintptr_t ma = mw4 & ~uintptr_t(15);
    if (oa < ob || oa + 16 * NVO > oe || ma < mb || ma + 16 * NVM > me) return false;
    words_from_window<NVO, NO>(orow, ow);
    words_from_window<NVM, NM>(reinterpret_cast<const void*>(mw4), mw);
    if constexpr (kEs == 2) {
      // the row starts in the upper half of its first word: shift by a half
      if (reinterpret_cast<uintptr_t>(mrow) & 2) {
#pragma unroll
        for (int i = 0; i < NM; ++i)
          mw[i] = __funnelshift_r(mw[i], i + 1 < NM ? mw[i + 1] : 0u, 16);
      }
    }
    return true;
  }
  // A merged 64-byte row (P = 9, 16-bit storage, row stride 32 elements,
  // 32-byte aligned): 2P offsets then P mask values read with two 256-bit
  // loads.  Offset pair p is word p; mask value p is half 18 + p, i.e. the
  // same words and halves as the separate mask row after its shift.
  __device__ __forceinline__ void load_merged64(const T* orow) {
    static_assert(KP == 9 && kEs == 2, "64-byte merged rows hold P = 9 16-bit rows");
    uint32_t w[16];
    ldg_words<16>(orow, w);
#pragma unroll
    for (int i = 0; i < NO; ++i) ow[i] = w[i];
#pragma unroll
    for (int i = 0; i < NM; ++i) mw[i] = w[NO + i];
  }
  __device__ __forceinline__ float2 off(int p) const {
    if constexpr (kEs == 2) {
      float f[2];
      Dt<T>::unpack(ow[p], f);
      return make_float2(f[0], f[1]);
    } else {
      return make_float2(__uint_as_float(ow[2 * p]), __uint_as_float(ow[2 * p + 1]));
    }
  }
  __device__ __forceinline__ float msk(int p) const {
    if constexpr (kEs == 2) {
      float f[2];
      Dt<T>::unpack(mw[p >> 1], f);
      return f[p & 1];
    } else {
      return __uint_as_float(mw[p]);
    }
  }
};

// v (NW words, NW/4 chunks of 16 bytes) rotated so that chunk j holds the
// former chunk (j + rot) mod NC; selects only, registers stay registers.
template <int NW>
__device__ __forceinline__ void rotate_chunks(uint32_t (&v)[NW], int rot) {
  constexpr int NC = NW / 4;
  if constexpr (NC > 1) {
    uint32_t o[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) o[i] = v[i];
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t x = o[4 * j + e];
#pragma unroll
        for (int r = 1; r < NC; ++r) x = rot == r ? o[4 * ((j + r) % NC) + e] : x;
        v[4 * j + e] = x;
      }
  }
}

// acc[0..2*NW) += weight * (the 16-bit or 32-bit elements packed in w), one
// product per element, accumulated in float32.  16-bit storage: the weight is
// rounded to the storage type once and each product is exact in float32
// (mixed-precision fma.rn.f32.{f16,bf16}); float32 storage: paired f32x2 FMAs.
template <typename T> struct Fma;

template <> struct Fma<__half> {
  using W = unsigned short;
  __device__ __forceinline__ static W weight(float w) {
    return __half_as_ushort(__float2half_rn(w));
  }
  __device__ __forceinline__ static void word(float& a0, float& a1, uint32_t v, W w) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.f16 %0, lo, %3, %0;\n\tfma.rn.f32.f16 %1, hi, %3, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(v), "h"(w));
  }
};

template <> struct Fma<__nv_bfloat16> {
  using W = unsigned short;
  __device__ __forceinline__ static W weight(float w) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(w));
  }
  __device__ __forceinline__ static void word(float& a0, float& a1, uint32_t v, W w) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.bf16 %0, lo, %3, %0;\n\tfma.rn.f32.bf16 %1, hi, %3, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(v), "h"(w));
  }
};

template <> struct Fma<float> {
  using W = float;
  __device__ __forceinline__ static W weight(float w) { return w; }
  // two consecutive float32 elements (words v0, v1) in one f32x2 FMA
  __device__ __forceinline__ static void pair(float& a0, float& a1, uint32_t v0, uint32_t v1,
                                              float w) {
    asm("{\n\t.reg .b64 a, c, s;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 c, {%2, %3};\n\t"
        "mov.b64 s, {%4, %4};\n\tfma.rn.f32x2 a, c, s, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(v0), "r"(v1), "f"(w));
  }
};

// s0 += lo(v) * lo(g), s1 += hi(v) * hi(g): the dot product of two packed
// 16-bit pairs, each product exact in float32.
template <typename T>
__device__ __forceinline__ void dot_word(float& s0, float& s1, uint32_t v, uint32_t g);

template <>
__device__ __forceinline__ void dot_word<__half>(float& s0, float& s1, uint32_t v, uint32_t g) {
  asm("{\n\t.reg .b16 vl, vh, gl, gh;\n\tmov.b32 {vl, vh}, %2;\n\tmov.b32 {gl, gh}, %3;\n\t"
      "fma.rn.f32.f16 %0, vl, gl, %0;\n\tfma.rn.f32.f16 %1, vh, gh, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(v), "r"(g));
}

template <>
__device__ __forceinline__ void dot_word<__nv_bfloat16>(float& s0, float& s1, uint32_t v,
                                                        uint32_t g) {
  asm("{\n\t.reg .b16 vl, vh, gl, gh;\n\tmov.b32 {vl, vh}, %2;\n\tmov.b32 {gl, gh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, vl, gl, %0;\n\tfma.rn.f32.bf16 %1, vh, gh, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(v), "r"(g));
}

// The 16-bit halves of the words of a grad_out slice, split once so that the
// dot products below split only the sampled words.
template <int NW>
struct Halves {
  unsigned short lo[NW], hi[NW];
  __device__ __forceinline__ void split(const uint32_t (&w)[NW]) {
#pragma unroll
    for (int i = 0; i < NW; ++i) asm("mov.b32 {%0, %1}, %2;" : "=h"(lo[i]), "=h"(hi[i]) : "r"(w[i]));
  }
};

// s0 += lo(v) * g0, s1 += hi(v) * g1: the dot product of a packed 16-bit pair
// with two grad_out halves already split, each product exact in float32.
template <typename T>
__device__ __forceinline__ void dot_split(float& s0, float& s1, uint32_t v, unsigned short g0,
                                          unsigned short g1);

template <>
__device__ __forceinline__ void dot_split<__half>(float& s0, float& s1, uint32_t v,
                                                  unsigned short g0, unsigned short g1) {
  asm("{\n\t.reg .b16 vl, vh;\n\tmov.b32 {vl, vh}, %2;\n\t"
      "fma.rn.f32.f16 %0, vl, %3, %0;\n\tfma.rn.f32.f16 %1, vh, %4, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(v), "h"(g0), "h"(g1));
}

template <>
__device__ __forceinline__ void dot_split<__nv_bfloat16>(float& s0, float& s1, uint32_t v,
                                                         unsigned short g0, unsigned short g1) {
  asm("{\n\t.reg .b16 vl, vh;\n\tmov.b32 {vl, vh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, vl, %3, %0;\n\tfma.rn.f32.bf16 %1, vh, %4, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(v), "h"(g0), "h"(g1));
}

template <typename T, int NW>
__device__ __forceinline__ void fma_words(float* acc, const uint32_t (&v)[NW], typename Fma<T>::W w) {
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int i = 0; i < NW; ++i) Fma<T>::word(acc[2 * i], acc[2 * i + 1], v[i], w);
  } else {
#pragma unroll
    for (int i = 0; i < NW; i += 2) Fma<T>::pair(acc[i], acc[i + 1], v[i], v[i + 1], w);
  }
}

// The shared-memory stride (elements of es bytes) of gradient rows of la
// elements staged one unit per lane: a row of an even number of 32-bit words
// gets one more word, so that consecutive lanes' rows start in different
// banks (64-byte merged rows otherwise put every second lane's store in the
// same bank).
__host__ __device__ inline int stage_stride(int la, int es) {
  return (la * es) % 4 == 0 && ((la * es) / 4) % 2 == 0 ? la + 4 / es : la;
}

// Copy `rows` rows of `row_bytes` (even) from shared memory rows `src_stride`
// bytes apart (even) to contiguous global memory over the lanes of one warp,
// in 32-bit words when the destination, the rows and the stride allow it,
// else in 16-bit halves.
template <typename U>
__device__ __forceinline__ void copy_rows_by(U* d, const U* s, int rows, int per_row, int stride,
                                             int lane) {
  for (int i = lane; i < rows * per_row; i += 32) {
    const int r = i / per_row;
    d[i] = s[r * stride + (i - r * per_row)];
  }
}
__device__ __forceinline__ void warp_copy_rows_out(void* dst, const void* src, int rows,
                                                   int row_bytes, int src_stride, int lane) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) |
                      static_cast<uintptr_t>(row_bytes) | static_cast<uintptr_t>(src_stride);
  if ((a & 3) == 0)
    copy_rows_by(static_cast<uint32_t*>(dst), static_cast<const uint32_t*>(src), rows,
                 row_bytes / 4, src_stride / 4, lane);
  else
    copy_rows_by(static_cast<unsigned short*>(dst), static_cast<const unsigned short*>(src), rows,
                 row_bytes / 2, src_stride / 2, lane);
}

// Copy `bytes` (even) from shared to global memory with the lanes of one warp,
// in 16-byte pieces when both ends and the length allow it.
__device__ __forceinline__ void warp_copy_out(void* dst, const void* src, int bytes, int lane) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) |
                      static_cast<uintptr_t>(bytes);
  if ((a & 15) == 0) {
    uint4* d = static_cast<uint4*>(dst);
    const uint4* s = static_cast<const uint4*>(src);
    for (int i = lane; i < bytes / 16; i += 32) d[i] = s[i];
  } else if ((a & 3) == 0) {
    uint32_t* d = static_cast<uint32_t*>(dst);
    const uint32_t* s = static_cast<const uint32_t*>(src);
    for (int i = lane; i < bytes / 4; i += 32) d[i] = s[i];
  } else {
    unsigned short* d = static_cast<unsigned short*>(dst);
    const unsigned short* s = static_cast<const unsigned short*>(src);
    for (int i = lane; i < bytes / 2; i += 32) d[i] = s[i];
  }
}

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
