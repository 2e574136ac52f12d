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
// linear_simt_kernel: any shape and float32, shared-memory tiles on the CUDA
// cores, float32 accumulation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"
#include "dcn_options.h"

namespace dcn {

__device__ unsigned long long g_linear_wait_timeouts = 0;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
constexpr int kLinearWaitPolls = 1 << 22;

// x (M, K), w (N, K) and y (M, N) through tensor maps with boxes of 64
// columns (128 bytes, 128-byte swizzle) by 128 rows (x, y) or N rows (w);
// K = 64 * KB, N a multiple of 16 up to 256 (the store clips the last block
// at N).  Dynamic shared memory: 1024 bytes of alignment slack, then
// KB x [128 x 128 B] of x and KB x [N x 128 B] of w (later the staging blocks
// of y), then two barriers and the tensor-memory address.
template <typename T>
__global__ void __launch_bounds__(128)
linear_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 const __grid_constant__ CUtensorMap ymap, int M, int N, int KB, int tcols,
                 const T* __restrict__ bias) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled layout is defined on 1024-byte aligned addresses
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* xs = smem;
  unsigned char* ws = smem + KB * 128 * 128;
  // after the MMAs the operand tiles are free: the output is staged there,
  // one 128-row x 64-column (128-byte) swizzled block per 64 outputs
  unsigned char* ys = smem;
  const int opnd = KB * (128 + N) * 128, stage = 128 * ((N + 63) / 64) * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (opnd > stage ? opnd : stage));
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
    // warp w holds rows 32w .. 32w + 31 of the tile in tensor-memory lanes;
    // each thread writes its row into the staging blocks (16-byte chunk j of
    // row r at chunk j ^ (r & 7), the layout the store's swizzle reads), then
    // one thread stores each 64-column block with a tensor copy, which clips
    // rows past M
    const int r = warp * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tbase + (uint32_t)c, v);
      if (bias) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += to_f32(bias[c + i]);
      }
      uint32_t wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wv[i] = Dt<T>::pack(v + 2 * i);
      unsigned char* blk = ys + (c >> 6) * (128 * 128) + r * 128;
      const int j0 = (c & 63) >> 3;  // first 16-byte chunk of these 16 columns
      *reinterpret_cast<uint4*>(blk + (((j0) ^ (r & 7)) << 4)) =
          make_uint4(wv[0], wv[1], wv[2], wv[3]);
      *reinterpret_cast<uint4*>(blk + (((j0 + 1) ^ (r & 7)) << 4)) =
          make_uint4(wv[4], wv[5], wv[6], wv[7]);
    }
    // the generic-proxy writes above become visible to the tensor copy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int c = 0; c < N; c += 64)
        asm volatile(
            "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::
                "l"(reinterpret_cast<uint64_t>(&ymap)),
            "r"(c), "r"(m0), "r"(smem_addr(ys + (c >> 6) * (128 * 128)))
            : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // the block's shared memory must outlive the copies' reads of it
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
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

// ---- the persistent, warp-specialised version ---------------------------------
// One CTA per SM walks the 128-row tiles t = blockIdx.x + i * gridDim.x:
//   warp 0 (one lane): the producer.  W once into shared memory, then the x
//     tiles into a ring of S stages (full / empty barriers per stage);
//   warp 1 (one lane): the MMA issuer.  Per tile, the tcgen05.mma chain into
//     one of two tensor-memory accumulators, then commits that free the x stage
//     and announce the accumulator;
//   warps 2-9: the epilogue.  Each reads a quarter of the accumulator's 128
//     lanes (warp w: lanes 32 * (w % 4) ...) for half of its columns, frees
//     the accumulator, adds the bias (staged once in shared memory), writes
//     the staging block of its buffer (two, alternating), and one thread
//     stores the tile with tensor copies while the next tile's MMAs run.
// All waits are bounded.  A role whose wait runs out raises the block's
// abort flag; the others see it in their own waits and stop; the epilogue
// warps decide together (a barrier reduction), so none is left at a barrier.
struct LinearWs {
  int S;          // x stages
  int ntiles;     // ceil(M / 128)
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort) {
  for (int i = 0; i < kLinearWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

template <typename T>
__global__ void __launch_bounds__(320, 1)
linear_ws_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 const __grid_constant__ CUtensorMap ymap, int N, int KB, int tcols, int S,
                 int YB, int ntiles, const T* __restrict__ bias) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int ystage = 128 * ((N + 63) / 64) * 128;  // one staging buffer
  unsigned char* ws = smem;                          // KB x N x 128 B
  unsigned char* as = ws + KB * N * 128;             // S x KB x 16 KB
  unsigned char* ys = as + S * KB * 128 * 128;       // YB x ystage (1 or 2)
  uint64_t* bars = reinterpret_cast<uint64_t*>(ys + YB * ystage);
  uint64_t* wfull = bars;                            // 1
  uint64_t* afull = bars + 1;                        // S
  uint64_t* aempty = afull + S;                      // S
  uint64_t* tfull = aempty + S;                      // 2
  uint64_t* tempty = tfull + 2;                      // 2
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  float* sbias = reinterpret_cast<float*>(tslot + 4);  // N
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(2 * tcols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    mbar_init(wfull, 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);
    }
    *abort = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // ---- producer
    mbar_expect_tx(wfull, (uint32_t)(KB * N * 128));
    for (int kb = 0; kb < KB; ++kb) tma_load_2d(ws + kb * N * 128, &wmap, wfull, kb * 64, 0);
    int i = 0, last = -1;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int st = i % S;
      if (!wait_or_abort(&aempty[st], ((i / S) & 1) ^ 1, abort)) break;
      mbar_expect_tx(&afull[st], (uint32_t)(KB * 128 * 128));
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d(as + (st * KB + kb) * 128 * 128, &xmap, &afull[st], kb * 64, t * 128);
      last = i;
    }
    if (*abort) {
      // leave no copy in flight into shared memory the next block may own:
      // W, and the latest copy into each stage (earlier ones completed before
      // their stage was refilled); every wait bounded
      mbar_wait_bounded(wfull, 0, kLinearWaitPolls);
      for (int j = last - S + 1 > 0 ? last - S + 1 : 0; j <= last; ++j)
        mbar_wait_bounded(&afull[j % S], (uint32_t)((j / S) & 1), kLinearWaitPolls);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = mma_idesc(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u,
                                     (uint32_t)N, 128u);
    int last = -1;
    if (wait_or_abort(wfull, 0, abort)) {
      int i = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
        const int st = i % S, b = i & 1;
        if (!wait_or_abort(&afull[st], (i / S) & 1, abort)) break;
        if (!wait_or_abort(&tempty[b], ((i >> 1) & 1) ^ 1, abort)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(b * tcols);
        for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sw128_desc(smem_addr(as + (st * KB + kb) * 128 * 128) + 32u * kk);
            const uint64_t bd = sw128_desc(smem_addr(ws + kb * N * 128) + 32u * kk);
            const uint32_t acc = (kb | kk) != 0;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
                : "memory");
          }
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&aempty[st]))
            : "memory");
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&tfull[b]))
            : "memory");
        last = i;
      }
    }
    // on abort, the MMAs already issued must finish before tensor memory is
    // freed: the last commit tracks all of them (bounded)
    if (*abort && last >= 0)
      mbar_wait_bounded(&tfull[last & 1], (uint32_t)((last >> 1) & 1), kLinearWaitPolls);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads tensor-memory lanes 32 * (w % 4) ... for the
    // columns of half (w - 2) / 4
    const int q = warp & 3, r = q * 32 + lane, half = (warp - 2) >> 2;
    const int et = threadIdx.x - 64;
    const bool leader = et == 0;
    const int c0 = half * (N >> 1), c1 = c0 + (N >> 1);
    for (int c = et; c < N; c += 256) sbias[c] = bias ? to_f32(bias[c]) : 0.f;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      const bool ok = wait_or_abort(&tfull[b], (i >> 1) & 1, abort);
      // all eight warps stop together if any wait ran out
      uint32_t bad;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(bad)
          : "r"(ok ? 0 : 1)
          : "memory");
      if (bad) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // the staging buffer was last stored YB tiles ago: its copy must have
      // read it (with two buffers the previous tile's copy may still read)
      if (leader && i >= YB) {
        if (YB == 2)
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        else
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      unsigned char* yb = ys + (YB == 2 ? b : 0) * ystage;
      const uint32_t tbase = tmem + (uint32_t)(b * tcols) + ((uint32_t)(q * 32) << 16);
      for (int c = c0; c < c1; c += 32) {
        // two loads in flight, one wait
        uint32_t ra[16], rb[16];
        tmem_ld16_async(tbase + (uint32_t)c, ra);
        tmem_ld16_async(tbase + (uint32_t)(c + 16), rb);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t* rr = hh ? rb : ra;
          const int cc = c + 16 * hh;
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(rr[e]) + sbias[cc + e];
          uint32_t wv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) wv[e] = Dt<T>::pack(v + 2 * e);
          unsigned char* blk = yb + (cc >> 6) * (128 * 128) + r * 128;
          const int j0 = (cc & 63) >> 3;
          *reinterpret_cast<uint4*>(blk + ((j0 ^ (r & 7)) << 4)) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(blk + (((j0 + 1) ^ (r & 7)) << 4)) =
              make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
      }
      // the accumulator is read: the MMA of tile i + 2 may overwrite it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (lane == 0) mbar_arrive(&tempty[b]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (leader) {
        for (int c = 0; c < N; c += 64)
          asm volatile(
              "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::
                  "l"(reinterpret_cast<uint64_t>(&ymap)),
              "r"(c), "r"(t * 128), "r"(smem_addr(yb + (c >> 6) * (128 * 128)))
              : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    if (leader) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && *abort) atomicAdd(&g_linear_wait_timeouts, 1ull);
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(2 * tcols)
                 : "memory");
  }
}

// ---- any K and N: the K loop through a ring of (x, W) chunk stages -----------
// The same roles as linear_ws_kernel, for layers whose W does not fit in
// shared memory (K > 256 or N > 256, e.g. InternImage-G's 512 -> 512
// projections).  Output tiles are 128 rows x BN columns (BN = 64, 128 or 256
// dividing N), walked n-tile fastest so that the tiles of one row block reuse
// its x chunks from L2.  Per tile the producer streams KB chunks of 64
// channels, each an x block (128 x 128 B) and a W block (BN x 128 B), through
// S stages; the MMA issuer consumes a stage with four K = 16 MMAs and frees it
// by a commit; the last chunk's commit announces the accumulator.
template <typename T>
__global__ void __launch_bounds__(320, 1)
linear_kloop_kernel(const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap ymap, int BN, int KB, int S, int YB,
                    int ntn, int ntiles, const T* __restrict__ bias, T* __restrict__ y, int M,
                    int N) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int abytes = 128 * 128, bbytes = BN * 128, sbytes = abytes + bbytes;
  const int ystage = 128 * BN * 2;                   // one staging buffer
  unsigned char* st_base = smem;                     // S x (x block, W block)
  unsigned char* ys = st_base + S * sbytes;          // YB x ystage
  uint64_t* bars = reinterpret_cast<uint64_t*>(ys + YB * ystage);
  uint64_t* afull = bars;                            // S
  uint64_t* aempty = afull + S;                      // S
  uint64_t* tfull = aempty + S;                      // 2
  uint64_t* tempty = tfull + 2;                      // 2
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  float* sbias = reinterpret_cast<float*>(tslot + 4);  // N
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);
    }
    *abort = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // ---- producer: chunk c of the CTA's sequence goes to stage c % S
    int c = 0;
    bool go = true;
    for (int t = blockIdx.x; go && t < ntiles; t += gridDim.x) {
      const int m0 = (t / ntn) * 128, n0 = (t % ntn) * BN;
      for (int kb = 0; kb < KB; ++kb, ++c) {
        const int st = c % S;
        if (!wait_or_abort(&aempty[st], ((c / S) & 1) ^ 1, abort)) {
          go = false;
          break;
        }
        unsigned char* a = st_base + st * sbytes;
        mbar_expect_tx(&afull[st], (uint32_t)sbytes);
        tma_load_2d(a, &xmap, &afull[st], kb * 64, m0);
        tma_load_2d(a + abytes, &wmap, &afull[st], kb * 64, n0);
      }
    }
    // no copy into this block's memory outlives it: wait (bounded) for the
    // last chunk issued into each stage (at once when the MMAs consumed it)
    for (int st = 0; st < S && st < c; ++st) {
      const int last = st + ((c - 1 - st) / S) * S;
      mbar_wait_bounded(&afull[st], (last / S) & 1, kLinearWaitPolls);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = mma_idesc(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u,
                                     (uint32_t)BN, 128u);
    int c = 0, i = 0;
    bool go = true;
    for (int t = blockIdx.x; go && t < ntiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      if (!wait_or_abort(&tempty[b], ((i >> 1) & 1) ^ 1, abort)) break;
      const uint32_t d = tmem + (uint32_t)(b * BN);
      for (int kb = 0; kb < KB; ++kb, ++c) {
        const int st = c % S;
        if (!wait_or_abort(&afull[st], (c / S) & 1, abort)) {
          go = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a = smem_addr(st_base + st * sbytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(a + 32u * kk);
          const uint64_t bd = sw128_desc(a + (uint32_t)abytes + 32u * kk);
          const uint32_t acc = (kb | kk) != 0;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
              "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&aempty[st]))
            : "memory");
      }
      if (!go) break;
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_addr(&tfull[b]))
          : "memory");
    }
    // the MMAs issued are complete before the tensor memory is freed: the
    // last commit tracks all of them (bounded)
    if (c > 0) mbar_wait_bounded(&aempty[(c - 1) % S], ((c - 1) / S) & 1, kLinearWaitPolls);
  } else if (warp >= 2) {
    // ---- epilogue, as in linear_ws_kernel, for a BN-column tile at n0
    const int q = warp & 3, r = q * 32 + lane, half = (warp - 2) >> 2;
    const bool leader = threadIdx.x == 64;
    const int c0 = half * (BN >> 1), c1 = c0 + (BN >> 1);
    for (int c = threadIdx.x - 64; c < N; c += 256) sbias[c] = bias ? to_f32(bias[c]) : 0.f;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int m0 = (t / ntn) * 128, n0 = (t % ntn) * BN;
      const int b = i & 1;
      const bool ok = wait_or_abort(&tfull[b], (i >> 1) & 1, abort);
      uint32_t bad;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(bad)
          : "r"(ok ? 0 : 1)
          : "memory");
      if (bad) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (leader && YB > 0 && i >= YB) {
        if (YB == 2)
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        else
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
      if (YB > 0) asm volatile("bar.sync 1, 256;" ::: "memory");
      unsigned char* yb = ys + (YB == 2 ? b : 0) * ystage;
      const uint32_t tbase = tmem + (uint32_t)(b * BN) + ((uint32_t)(q * 32) << 16);
      T* yrow = y + (size_t)(m0 + r) * N + n0;  // YB == 0: this thread's row
      for (int c = c0; c < c1; c += 32) {
        uint32_t ra[16], rb[16];
        tmem_ld16_async(tbase + (uint32_t)c, ra);
        tmem_ld16_async(tbase + (uint32_t)(c + 16), rb);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t* rr = hh ? rb : ra;
          const int cc = c + 16 * hh;
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            v[e] = __uint_as_float(rr[e]) + sbias[n0 + cc + e];
          uint32_t wv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) wv[e] = Dt<T>::pack(v + 2 * e);
          if (YB == 0) {
            // straight to memory: 32 contiguous bytes of the row, rows past M
            // skipped
            if (m0 + r < M) {
              uint4* dst = reinterpret_cast<uint4*>(yrow + cc);
              dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
              dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            }
          } else {
            unsigned char* blk = yb + (cc >> 6) * (128 * 128) + r * 128;
            const int j0 = (cc & 63) >> 3;
            *reinterpret_cast<uint4*>(blk + ((j0 ^ (r & 7)) << 4)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
            *reinterpret_cast<uint4*>(blk + (((j0 + 1) ^ (r & 7)) << 4)) =
                make_uint4(wv[4], wv[5], wv[6], wv[7]);
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (lane == 0) mbar_arrive(&tempty[b]);
      if (YB == 0) continue;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (leader) {
        for (int c = 0; c < BN; c += 64)
          asm volatile(
              "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::
                  "l"(reinterpret_cast<uint64_t>(&ymap)),
              "r"(n0 + c), "r"(m0), "r"(smem_addr(yb + (c >> 6) * (128 * 128)))
              : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    if (leader && YB > 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && *abort) atomicAdd(&g_linear_wait_timeouts, 1ull);
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(2 * BN)
                 : "memory");
  }
}

// Any shape, any of the three types: 64 x 64 output tiles per block of 256
// threads (4 x 4 outputs each), the x and W slices of 32 channels staged in
// shared memory, float32 accumulation.
template <typename T>
__global__ void __launch_bounds__(256)
linear_simt_kernel(const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ bias,
                   T* __restrict__ y, long long M, int K, int N) {
  __shared__ float xs[32][65];
  __shared__ float wsh[32][65];
  const long long m0 = (long long)blockIdx.x * 64;
  const int n0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int rr = i >> 5, kk = i & 31;
      const long long m = m0 + rr;
      const int n = n0 + rr, k = k0 + kk;
      xs[kk][rr] = (m < M && k < K) ? to_f32(x[m * K + k]) : 0.f;
      wsh[kk][rr] = (n < N && k < K) ? to_f32(w[(size_t)n * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = xs[kk][ty * 4 + i];
        bb[i] = wsh[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) y[m * N + n] = Dt<T>::from_f(acc[i][j] + (bias ? to_f32(bias[n]) : 0.f));
    }
  }
}

// ---- host side ------------------------------------------------------------------

static int dev_of_stream() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

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

// Shared memory of the persistent kernel with S x stages and YB output
// staging buffers (two if they fit, else one; 0 when not even S = 2, YB = 1
// fits in 227 KB).
static size_t linear_ws_smem(int K, int N, int* S_out, int* YB_out, size_t budget = 227 * 1024) {
  const size_t KB = K / 64, w = KB * N * 128, a = KB * 128 * 128,
               y = (size_t)128 * ((N + 63) / 64) * 128,
               bars = 8 * (1 + 2 * 4 + 4) + 16 + 4 * (size_t)N;
  for (int YB = 2; YB >= 1; --YB)
    for (int S = 4; S >= 2; --S) {
      const size_t total = 1024 + w + S * a + YB * y + bars;
      if (total <= budget) {
        *S_out = S;
        *YB_out = YB;
        return total;
      }
    }
  return 0;
}

// The K-loop kernel's output tile width: 256, 128 or 64 columns dividing N
// (the linear_bn switch caps it).
static int linear_kloop_bn(int N) {
  const int cap = options().linear_bn;
  for (int bn = 256; bn >= 64; bn >>= 1)
    if (bn <= cap && N % bn == 0) return bn;
  return 0;
}

// Shared memory of the K-loop kernel: S stages of (x, W) chunks, YB output
// staging buffers and the bias, the deepest pipeline first.  YB = 0 (rows
// stored straight from registers, the linear_yb switch at 0) frees the staging memory
// for stages but measured slower (131072 x 512 -> 512: 96 us against 82 us).
static size_t linear_kloop_smem(int BN, int N, int* S_out, int* YB_out) {
  const size_t sb = (size_t)(128 + BN) * 128, y = (size_t)128 * BN * 2;
  const int ybmax = options().linear_yb, smax = options().linear_s;
  const int ybmin = ybmax == 0 ? 0 : 1;
  for (int S = smax; S >= 2; --S)
    for (int YB = ybmax; YB >= ybmin; --YB) {
      const size_t total = 1024 + S * sb + YB * y + 8 * (2 * S + 4) + 16 + 4 * (size_t)N;
      if (total <= 227 * 1024) {
        *S_out = S;
        *YB_out = YB;
        return total;
      }
    }
  return 0;
}

size_t linear_tc_smem(int K, int N) {
  const size_t opnd = (size_t)(K / 64) * (128 + N) * 128,
               stage = (size_t)128 * ((N + 63) / 64) * 128;
  return 1024 + (opnd > stage ? opnd : stage) + 32;
}

bool linear_tc_ok(int dtype, long long M, int K, int N, const void* x, const void* w,
                  const void* y) {
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!(dtype == DCN_F16 || dtype == DCN_BF16) || M < 1 || K % 64 || K < 64 || N % 16 ||
      N < 16 || !a16(x) || !a16(w) || !a16(y) || M > (long long)INT_MAX - 128 ||
      linear_encoder() == nullptr)
    return false;
  if (K <= 256 && N <= 256) return linear_tc_smem(K, N) <= 200 * 1024;
  // the K-loop kernel: whole 64-column output blocks, tiles counted in int
  const int bn = linear_kloop_bn(N);
  int S = 0, YB = 0;
  return bn > 0 && (M + 127) / 128 * (N / bn) <= INT_MAX &&
         linear_kloop_smem(bn, N, &S, &YB) != 0;
}

template <typename T>
static cudaError_t launch_linear_t(int dtype, long long M, int K, int N, const void* x,
                                   const void* w, const void* b, void* y, bool tc,
                                   cudaStream_t s) {
  const T* b_ = static_cast<const T*>(b);
  T* y_ = static_cast<T*>(y);
  if constexpr (sizeof(T) == 2) {
    if (tc && (K > 256 || N > 256)) {
      const int BN = linear_kloop_bn(N);
      int S = 0, YB = 0;
      const size_t smem = BN ? linear_kloop_smem(BN, N, &S, &YB) : 0;
      if (!smem) return cudaErrorInvalidValue;
      CUtensorMap xm, wm, ym;
      if (!encode_rows(&xm, dtype, x, M, K, 128) || !encode_rows(&wm, dtype, w, N, K, BN) ||
          !encode_rows(&ym, dtype, y, M, N, 128))
        return cudaErrorInvalidValue;
      cudaError_t e = cudaFuncSetAttribute(linear_kloop_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_of_stream());
      if (e != cudaSuccess) return e;
      const int ntn = N / BN;
      const int ntiles = (int)((M + 127) / 128) * ntn;
      const int grid = ntiles < sms ? ntiles : sms;
      linear_kloop_kernel<T><<<grid, 320, smem, s>>>(xm, wm, ym, BN, K / 64, S, YB, ntn, ntiles,
                                                     b_, y_, (int)M, N);
      return cudaGetLastError();
    }
    if (tc) {
      CUtensorMap xm, wm, ym;
      if (!encode_rows(&xm, dtype, x, M, K, 128) || !encode_rows(&wm, dtype, w, N, K, N) ||
          !encode_rows(&ym, dtype, y, M, N, 128))
        return cudaErrorInvalidValue;
      int tcols = 32;
      while (tcols < N) tcols <<= 1;
      int S = 0, YB = 0;
      // CTAs per SM: two when both fit (shared memory and 2 x 2 x tcols
      // tensor-memory columns), so that one CTA's epilogue overlaps the other's
      int per_sm = options().linear_ctas >= 2 && 4 * tcols <= 512 ? 2 : 1;
      size_t wsm = linear_ws_smem(K, N, &S, &YB, per_sm == 2 ? 113 * 1024 : 227 * 1024);
      if (!wsm && per_sm == 2) {
        per_sm = 1;
        wsm = linear_ws_smem(K, N, &S, &YB);
      }
      if (wsm && 2 * tcols <= 512 && N % 64 == 0 && options().linear_persist) {
        cudaError_t e = cudaFuncSetAttribute(linear_ws_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_of_stream());
        if (e != cudaSuccess) return e;
        const int ntiles = (int)((M + 127) / 128);
        const int grid = ntiles < per_sm * sms ? ntiles : per_sm * sms;
        linear_ws_kernel<T><<<grid, 320, wsm, s>>>(xm, wm, ym, N, K / 64, tcols, S, YB, ntiles,
                                                   b_);
        return cudaGetLastError();
      }
      const size_t smem = linear_tc_smem(K, N);
      cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      const unsigned grid = (unsigned)((M + 127) / 128);
      linear_tc_kernel<T><<<grid, 128, smem, s>>>(xm, wm, ym, (int)M, N, K / 64, tcols, b_);
      return cudaGetLastError();
    }
  }
  const long long gx = (M + 63) / 64, gy = (N + 63) / 64;
  if (gx > INT_MAX || gy > 65535) return cudaErrorInvalidConfiguration;
  linear_simt_kernel<T><<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(
      static_cast<const T*>(x), static_cast<const T*>(w), b_, y_, M, K, N);
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
