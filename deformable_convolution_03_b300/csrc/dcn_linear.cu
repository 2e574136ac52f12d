// dcn_linear.cu -- the linear projections around the core op on the tensor
// cores: y = x W^T + b over the rows of a channels-last tensor.
//
// The DCN module feeds the core op through dense layers: DCNv3 projects the
// input, predicts offsets and mask logits with linear layers and projects the
// core's output (page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现
// 逐行解读", section 三, items 1-6); DCNv4 merges the offset and mask layers
// into one whose output is the merged offset/mask tensor (page "告别DCNv3的卡顿：
// 实测DCNv4在A100上3倍提速，手把手教你集成到FlashInternImage", section 1).
//
// linear_tc_kernel: one CTA of four warps per 128 rows.  Tensor copies (TMA)
// bring the block's rows of x and all of W, 64 channels per copy, into shared
// memory in the 128-byte-swizzled K-major layout; one thread issues the
// tcgen05.mma instructions (M = 128, N = the layer's outputs, K = 16 each),
// accumulating in float32 in tensor memory; each warp then reads its 32 rows
// of the accumulator with tcgen05.ld, adds the bias and stores its rows in
// the storage type.  Every wait is bounded: a block whose copy or MMA does
// not complete counts it (dcn_wait_timeouts), writes nothing, still frees its
// tensor memory and waits once more (bounded) for what it issued.
//
// linear_simt_kernel: any shape and float32, one thread per output element,
// float32 accumulation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>
#include <type_traits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {

__device__ unsigned long long g_linear_wait_timeouts = 0;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
constexpr int kLinearWaitPolls = 1 << 22;

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

// x (M, K) and w (N, K) through the tensor maps (boxes of 64 x 128 rows and
// 64 x N rows, 128-byte swizzle); K = 64 * KB, 16 <= N <= 256, N % 16 == 0.
// Dynamic shared memory: 1024 bytes of alignment slack, KB x [128 x 128 B] of
// x, KB x [N x 128 B] of w, then two barriers and the tensor-memory address.
template <typename T>
__global__ void __launch_bounds__(128)
linear_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 int M, int N, int KB, int tcols, const T* __restrict__ bias, T* __restrict__ y) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled layout is defined on 1024-byte aligned addresses
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* xs = smem;
  unsigned char* ws = smem + KB * 128 * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ws + KB * N * 128);  // [0] copies, [1] MMA
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(tcols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;

  bool ok = true, issued = false;
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bars[0], (uint32_t)(KB * (128 + N) * 128));
    for (int kb = 0; kb < KB; ++kb) {
      tma_load_2d(xs + kb * 128 * 128, &xmap, &bars[0], kb * 64, m0);
      tma_load_2d(ws + kb * N * 128, &wmap, &bars[0], kb * 64, 0);
    }
    ok = mbar_wait_bounded(&bars[0], 0, kLinearWaitPolls);
    if (ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t idesc = mma_idesc(sizeof(T) == 2 && !std::is_same<T, __half>::value ? 1u : 0u,
                                       (uint32_t)N, 128u);
      for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // the kk-th 16-element (32-byte) slice of the 128-byte rows
          const uint64_t ad = sw128_desc(smem_addr(xs + kb * 128 * 128) + 32u * kk);
          const uint64_t bd = sw128_desc(smem_addr(ws + kb * N * 128) + 32u * kk);
          const uint32_t acc = (kb | kk) != 0;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
              : "memory");
        }
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_addr(&bars[1]))
          : "memory");
      issued = true;
    }
  }
  // everyone learns whether the copies arrived, then waits for the MMAs
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (ok) ok = mbar_wait_bounded(&bars[1], 0, kLinearWaitPolls);
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (ok) {
    // warp w holds rows 32w .. 32w + 31 of the tile in tensor-memory lanes
    const int row = m0 + warp * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tbase + (uint32_t)c, v);
      if (bias) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += to_f32(bias[c + i]);
      }
      if (row < M) {
        uint32_t wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = Dt<T>::pack(v + 2 * i);
        uint4* dst = reinterpret_cast<uint4*>(y + (size_t)row * N + c);
        dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
      }
    }
  } else if (threadIdx.x == 0) {
    atomicAdd(&g_linear_wait_timeouts, 1ull);
    // leave nothing in flight: the copies, then the MMAs if they were issued
    // (both bounded)
    mbar_wait_bounded(&bars[0], 0, kLinearWaitPolls);
    if (issued) mbar_wait_bounded(&bars[1], 0, kLinearWaitPolls);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols)
                 : "memory");
  }
}

// Any shape, any of the three types: one thread per output element.
template <typename T>
__global__ void __launch_bounds__(256)
linear_simt_kernel(const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ bias,
                   T* __restrict__ y, long long M, int K, int N) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M * N) return;
  const long long m = i / N;
  const int n = (int)(i - m * N);
  const T* xr = x + m * K;
  const T* wr = w + (size_t)n * K;
  float acc = bias ? to_f32(bias[n]) : 0.f;
  for (int k = 0; k < K; ++k) acc = fmaf(to_f32(xr[k]), to_f32(wr[k]), acc);
  y[i] = Dt<T>::from_f(acc);
}

// ---- host side ------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 linear_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// a (rows x K) row-major 16-bit matrix, boxes of 64 x box_rows, 128-byte swizzle
static bool encode_rows(CUtensorMap* m, int dtype, const void* base, long long rows, int K,
                        int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = linear_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      dtype == DCN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t linear_tc_smem(int K, int N) { return 1024 + (size_t)(K / 64) * (128 + N) * 128 + 32; }

bool linear_tc_ok(int dtype, long long M, int K, int N, const void* x, const void* w,
                  const void* y) {
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return (dtype == DCN_F16 || dtype == DCN_BF16) && M >= 1 && K % 64 == 0 && K >= 64 &&
         K <= 256 && N % 16 == 0 && N >= 16 && N <= 256 && a16(x) && a16(w) && a16(y) &&
         M <= (long long)INT_MAX - 128 && linear_tc_smem(K, N) <= 200 * 1024 &&
         linear_encoder() != nullptr;
}

template <typename T>
static cudaError_t launch_linear_t(int dtype, long long M, int K, int N, const void* x,
                                   const void* w, const void* b, void* y, bool tc,
                                   cudaStream_t s) {
  const T* b_ = static_cast<const T*>(b);
  T* y_ = static_cast<T*>(y);
  if constexpr (sizeof(T) == 2) {
    if (tc) {
      CUtensorMap xm, wm;
      if (!encode_rows(&xm, dtype, x, M, K, 128) || !encode_rows(&wm, dtype, w, N, K, N))
        return cudaErrorInvalidValue;
      int tcols = 32;
      while (tcols < N) tcols <<= 1;
      const size_t smem = linear_tc_smem(K, N);
      cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      const unsigned grid = (unsigned)((M + 127) / 128);
      linear_tc_kernel<T><<<grid, 128, smem, s>>>(xm, wm, (int)M, N, K / 64, tcols, b_, y_);
      return cudaGetLastError();
    }
  }
  const long long total = M * N;
  const long long grid = (total + 255) / 256;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  linear_simt_kernel<T><<<(unsigned)grid, 256, 0, s>>>(static_cast<const T*>(x),
                                                       static_cast<const T*>(w), b_, y_, M, K, N);
  return cudaGetLastError();
}

cudaError_t launch_linear(int dtype, long long M, int K, int N, const void* x, const void* w,
                          const void* b, void* y, bool tc, cudaStream_t s) {
  switch (dtype) {
    case DCN_F32: return launch_linear_t<float>(dtype, M, K, N, x, w, b, y, false, s);
    case DCN_F16: return launch_linear_t<__half>(dtype, M, K, N, x, w, b, y, tc, s);
    case DCN_BF16: return launch_linear_t<__nv_bfloat16>(dtype, M, K, N, x, w, b, y, tc, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t read_linear_wait_timeouts(unsigned long long* count) {
  return cudaMemcpyFromSymbol(count, g_linear_wait_timeouts, sizeof(unsigned long long));
}

}  // namespace dcn
