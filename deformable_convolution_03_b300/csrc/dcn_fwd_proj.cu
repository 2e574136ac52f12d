// dcn_fwd_proj.cu -- DCNv4's forward with its merged offset/mask projection
// computed in the same launch.
//
// In the DCN module the offsets and the mask are linear projections of the
// control features x1 (page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现
// 逐行解读", section 三 items 3-4), and DCNv4 merges the two layers into one
// whose output rows hold a (pixel, group)'s 2P offsets, P mask values and
// padding (page "告别DCNv3的卡顿：实测DCNv4在A100上3倍提速，手把手教你集成到
// FlashInternImage", section 1).  Run separately, that layer writes the merged
// rows to memory and the core reads them back.  Here a block of the TMA-staged
// forward (dcn_fwd_tma.cu: a tile of output pixels for GB groups, the input
// window in shared memory) first computes its tile's rows on the tensor cores
// and keeps them in shared memory:
//   - one thread issues three tensor copies: the input window, the tile's
//     feature rows (a box of the (N, Ho, Wo, K) features, K-major, 128-byte
//     swizzle: row r = tile pixel r) and the block's GB * row_stride weight
//     rows, then the tcgen05.mma chain M = 128 (rows past the tile's pixels
//     are not used), N = GB * row_stride, K = 16 per instruction, float32
//     accumulation in tensor memory;
//   - warps 0-3 read the accumulator rows of the tile's pixels (tcgen05.ld),
//     add the bias and round to the storage type -- the same sum and the same
//     rounding as dcn_linear -- and write the rows into shared memory (and to
//     the merged offset/mask tensor when the caller passes one, for the
//     backward);
//   - the sampling threads then take their offsets and masks from shared
//     memory and run the forward's sampling loop unchanged.
// Every wait is bounded.  A block whose copy or MMA does not complete counts
// it (dcn_wait_timeouts), computes nothing, waits once more (bounded) for what
// it issued and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {

namespace {

__device__ unsigned long long g_proj_wait_timeouts = 0;
constexpr int kProjWaitPolls = 1 << 22;

// The inverse rotation of the accumulator chunks (see dcn_fwd_tma.cu).
template <int CPT, typename T>
__device__ __forceinline__ void unrotate(float (&acc)[CPT], int rot) {
  constexpr int PER = 16 / (int)sizeof(T);
  constexpr int NC = CPT / PER;
  if constexpr (NC > 1) {
    float o[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) o[i] = acc[i];
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        float x = o[PER * c + e];
#pragma unroll
        for (int r = 1; r < NC; ++r) x = rot == r ? o[PER * ((c - r + NC) % NC) + e] : x;
        acc[PER * c + e] = x;
      }
  }
}

// The forward over one tile, its offsets and masks taken from the rows in
// shared memory and its corners from the staged window (ready) or, for cells
// outside the window, from global memory.  tid: the thread's index among the
// block's sampling threads.
template <typename T, int CPT, int KP, int RB>
__device__ __forceinline__ void sample_tile(const KParams& kp, const TileGeom& tg,
                                            const ProjGeom& pg, int tid, int n, int gb, int ho0,
                                            int wo0, int wy0, int wx0, const T* oms,
                                            const unsigned char* win, bool ready,
                                            const T* __restrict__ input, T* __restrict__ output) {
  constexpr int NW = CPT * (int)sizeof(T) / 4;
  constexpr int NC = NW / 4;
  const int chunks = kp.gc / CPT;
  const int npx = kp.tile_w * kp.tile_h;
  const int rs = pg.rs;
  const int per_px = tg.GB * chunks;
  const int lp = tid / per_px, rr = tid - lp * per_px;
  const int gl = rr / chunks, slice = rr - gl * chunks;
  const int g = gb * tg.GB + gl, c0 = slice * CPT;
  const int ho = ho0 + lp / kp.tile_w, wo = wo0 + lp % kp.tile_w;
  const bool active = lp < npx && ho < kp.Ho && wo < kp.Wo;
  const size_t unit = active ? (((size_t)n * kp.Ho + ho) * kp.Wo + wo) * kp.G + g : 0;
  const int P = KP > 0 ? KP : kp.P;
  // this (pixel, group)'s row: 2P offsets, then P mask values
  const T* row = oms + (active ? lp : 0) * pg.om_stride + gl * rs;
  const T* img = input + (size_t)n * kp.H * kp.W * kp.C + g * kp.gc + c0;
  const uint32_t W = kp.W, H = kp.H, C = kp.C, WC = (uint32_t)kp.W * kp.C;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) {
    mx = -INFINITY;
    for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::to_f(row[2 * P + p]));
    float s = 0.f;
    for (int p = 0; p < P; ++p) s += expf(Dt<T>::to_f(row[2 * P + p]) - mx);
    inv = 1.f / s;
  }

  if (active) {
    float acc[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) acc[i] = 0.f;
    const uint32_t rb = RB > 0 ? (uint32_t)RB : (uint32_t)(tg.GB * kp.gc) * (uint32_t)sizeof(T);
    const uint32_t wrb = (uint32_t)tg.WW * rb;
    const uint32_t chunk0 = (uint32_t)(gl * kp.gc + c0) * (uint32_t)sizeof(T) / 16u;
    const int rot = NC > 1 ? lp & (NC - 1) : 0;
    uint32_t coff[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) coff[j] = 16u * (chunk0 + (uint32_t)((j + rot) & (NC - 1)));
    const int WWm = tg.WW - 1, WHm = tg.WH - 1;

    unsigned long long far = 0ull;
#pragma unroll(KP > 0 ? KP : 1)
    for (int p = 0; p < P; ++p) {
      float m = Dt<T>::to_f(row[2 * P + p]);
      const float dx = Dt<T>::to_f(row[2 * p]), dy = Dt<T>::to_f(row[2 * p + 1]);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float x = location(dx, kp.tap_x[p], scale, ref_x);
      const float y = location(dy, kp.tap_y[p], scale, ref_y);
      if (!in_box(x, y, kp.W, kp.H)) continue;  // also NaN / inf
      const float xf = floorf(x), yf = floorf(y);
      const int cx = (int)xf - wx0, cy = (int)yf - wy0;
      if (!(ready && (unsigned)cx < (unsigned)WWm && (unsigned)cy < (unsigned)WHm)) {
        far |= 1ull << p;
        continue;
      }
      const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
      const float gym = gy * m, fym = fy * m;
      const unsigned char* a00 = win + (uint32_t)(cy * tg.WW + cx) * rb;
      const uint32_t at[4] = {0u, rb, wrb, wrb + rb};
      const float w[4] = {gym * gx, gym * fx, fym * gx, fym * fx};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t v[NW];
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const unsigned char* q = a00 + coff[j] + at[k];
          const uint4 c = DCN_IN_SPAN(q, 16, win, tg.win_bytes, kBadShared)
                              ? *reinterpret_cast<const uint4*>(q)
                              : make_uint4(0u, 0u, 0u, 0u);
          v[4 * j] = c.x;
          v[4 * j + 1] = c.y;
          v[4 * j + 2] = c.z;
          v[4 * j + 3] = c.w;
        }
        fma_words<T, NW>(acc, v, Fma<T>::weight(w[k]));
      }
    }
    // far points: clamped corners from global memory, weight 0 outside
    while (far) {
      const int p = __ffsll((long long)far) - 1;
      far &= far - 1;
      float m = Dt<T>::to_f(row[2 * P + p]);
      const float dx = Dt<T>::to_f(row[2 * p]), dy = Dt<T>::to_f(row[2 * p + 1]);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float x = location(dx, kp.tap_x[p], scale, ref_x);
      const float y = location(dy, kp.tap_y[p], scale, ref_y);
      const float xf = floorf(x), yf = floorf(y);
      const int x0 = (int)xf, y0 = (int)yf;
      const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
      const float wy0v = (uint32_t)y0 < H ? gy * m : 0.f;
      const float wy1v = (uint32_t)(y0 + 1) < H ? fy * m : 0.f;
      const float wx0v = (uint32_t)x0 < W ? gx : 0.f;
      const float wx1v = (uint32_t)(x0 + 1) < W ? fx : 0.f;
      const uint32_t xa = min((uint32_t)x0, W - 1), xb = min((uint32_t)(x0 + 1), W - 1);
      const uint32_t ya = min((uint32_t)y0, H - 1), yb = min((uint32_t)(y0 + 1), H - 1);
      const uint32_t ra = ya * WC, rbb = yb * WC, ca = xa * C, cb = xb * C;
      uint32_t v00[NW], v01[NW], v10[NW], v11[NW];
      ldg_words_in<NW>(img + (ra + ca), v00, input, input_bytes<T>(kp));
      ldg_words_in<NW>(img + (ra + cb), v01, input, input_bytes<T>(kp));
      ldg_words_in<NW>(img + (rbb + ca), v10, input, input_bytes<T>(kp));
      ldg_words_in<NW>(img + (rbb + cb), v11, input, input_bytes<T>(kp));
      rotate_chunks<NW>(v00, rot);
      rotate_chunks<NW>(v01, rot);
      rotate_chunks<NW>(v10, rot);
      rotate_chunks<NW>(v11, rot);
      fma_words<T, NW>(acc, v00, Fma<T>::weight(wy0v * wx0v));
      fma_words<T, NW>(acc, v01, Fma<T>::weight(wy0v * wx1v));
      fma_words<T, NW>(acc, v10, Fma<T>::weight(wy1v * wx0v));
      fma_words<T, NW>(acc, v11, Fma<T>::weight(wy1v * wx1v));
    }
    unrotate<CPT, T>(acc, rot);
    if (out_in(kp, output, output + unit * kp.gc + c0, CPT))
      Slice<T, CPT>::store(output + unit * kp.gc + c0, acc);
  }
}

// RB as in fwd_tile_kernel: the bytes of a window pixel when 128, else 0.
template <typename T, int CPT, int KP, int RB>
__global__ void __launch_bounds__(256)
fwd_proj_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap fmap,
                const __grid_constant__ CUtensorMap wmap, const KParams kp, const TileGeom tg,
                const ProjGeom pg, const T* __restrict__ input, const T* __restrict__ bias,
                T* __restrict__ output, T* __restrict__ om_out) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled operand layout is defined on 1024-byte aligned addresses
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* win = smem + pg.win_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pg.bar_off);  // window, operands, MMA
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  T* oms = reinterpret_cast<T*>(smem);  // the rows, over the operands once the MMAs are done
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npx = kp.tile_w * kp.tile_h;
  const int NB = pg.NB, rs = pg.rs;

  // block -> (image, tile, group block), the group block fastest
  const int gb = blockIdx.x % tg.ngb;
  const int rest = blockIdx.x / tg.ngb;
  const int tiles = kp.tiles_w * kp.tiles_h;
  const int t = rest % tiles, n = rest / tiles;
  const int ty = t / kp.tiles_w;
  const int ho0 = ty * kp.tile_h, wo0 = (t - ty * kp.tiles_w) * kp.tile_w;
  const int wy0 = ho0 * kp.stride_h + tg.org_y, wx0 = wo0 * kp.stride_w + tg.org_x;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(pg.ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;

  // ---- the tile's offset/mask rows on the tensor cores ---------------------
  bool ok = true, issued = false;
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bars[0], tg.win_bytes);
    tma_load_4d(win, &tmap, &bars[0], gb * tg.GB * kp.gc, wx0, wy0, n);
    mbar_expect_tx(&bars[1], (uint32_t)(pg.KB * (npx + NB) * 128));
    for (int kb = 0; kb < pg.KB; ++kb) {
      tma_load_4d(smem + kb * 128 * 128, &fmap, &bars[1], kb * 64, wo0, ho0, n);
      tma_load_2d(smem + pg.b_off + kb * NB * 128, &wmap, &bars[1], kb * 64, gb * NB);
    }
    ok = mbar_wait_bounded(&bars[1], 0, kProjWaitPolls);
    if (ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t idesc = mma_idesc(std::is_same<T, __half>::value ? 0u : 1u, (uint32_t)NB,
                                       128u);
      for (int kb = 0; kb < pg.KB; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(smem_addr(smem + kb * 128 * 128) + 32u * kk);
          const uint64_t bd = sw128_desc(smem_addr(smem + pg.b_off + kb * NB * 128) + 32u * kk);
          const uint32_t accum = (kb | kk) != 0;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
              : "memory");
        }
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_addr(&bars[2]))
          : "memory");
      issued = true;
    }
  }
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (ok) ok = mbar_wait_bounded(&bars[2], 0, kProjWaitPolls);
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (!ok && threadIdx.x == 0) {
    atomicAdd(&g_proj_wait_timeouts, 1ull);
    // nothing may still write this block's memory when it goes on
    mbar_wait_bounded(&bars[1], 0, kProjWaitPolls);
    if (issued) mbar_wait_bounded(&bars[2], 0, kProjWaitPolls);
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (ok && warp < 4) {
    // warp w reads tensor-memory lanes 32w .. 32w + 31: tile pixels
    const int r = warp * 32 + lane;
    const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16);
    const int ho = ho0 + r / kp.tile_w, wo = wo0 + r % kp.tile_w;
    T* og = nullptr;
    if (om_out && r < npx && ho < kp.Ho && wo < kp.Wo)
      og = om_out + (((size_t)n * kp.Ho + ho) * kp.Wo + wo) * ((size_t)kp.G * rs) + gb * NB;
    T* os = oms + r * pg.om_stride;
    for (int c = 0; c < NB; c += 16) {
      float v[16];
      tmem_ld16(tb + (uint32_t)c, v);  // every lane of the warp takes part
      if (r >= npx) continue;
      if (bias) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += Dt<T>::to_f(bias[gb * NB + c + i]);
      }
      uint32_t wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wv[i] = Dt<T>::pack(v + 2 * i);
      const uint4 lo = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      const uint4 hi = make_uint4(wv[4], wv[5], wv[6], wv[7]);
      if (DCN_IN_SPAN(os + c, 32, smem, pg.om_bytes, kBadShared)) {
        reinterpret_cast<uint4*>(os + c)[0] = lo;
        reinterpret_cast<uint4*>(os + c)[1] = hi;
      }
      if (og) {
        reinterpret_cast<uint4*>(og + c)[0] = lo;
        reinterpret_cast<uint4*>(og + c)[1] = hi;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // the rows are in shared memory; tensor memory is read
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(pg.ncols)
                 : "memory");
  }

  // ---- the forward over the tile, offsets and masks from shared memory -----
  const bool ready = mbar_wait_bounded(&bars[0], 0, kProjWaitPolls);
  if (!ready && threadIdx.x == 0 && ok) atomicAdd(&g_proj_wait_timeouts, 1ull);
  if (ok)
    sample_tile<T, CPT, KP, RB>(kp, tg, pg, threadIdx.x, n, gb, ho0, wo0, wy0, wx0, oms, win,
                                ready, input, output);
  // a block whose wait ran out leaves no copy in flight into its memory
  if (!ready) mbar_wait_bounded(&bars[0], 0, kProjWaitPolls);
}

// A wait on an mbarrier that gives up when the block's abort flag is raised
// (checked every 256 polls) or after kProjWaitPolls polls (then raising it).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort) {
  for (int i = 0; i < kProjWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  return false;
}

// The persistent, warp-specialised version: one block per SM walks the tiles
// t = blockIdx.x + i * gridDim.x (gridDim.x a multiple of the group-block
// count, so a block always projects the same group block's rows and keeps
// their weights in shared memory).  Warps by role:
//   0 .. sw-1   sampling: wait for tile i's rows and window, run the forward
//               over the tile, release both (one arrival per warp);
//   sw          producer: the weights once, then per tile the window into one
//               of two window buffers and the feature rows into one of S
//               stages, each after its buffer was released;
//   sw+1        MMA issuer: per tile the tcgen05.mma chain into one of two
//               tensor-memory accumulators, committing to free the feature
//               stage and to announce the accumulator;
//   sw+2..sw+5  rows: per tile read the accumulator (each warp its lane
//               quarter), add the bias, round, write one of two row buffers
//               (and offset_mask when given), release the accumulator and
//               announce the rows.
// So the projection of tile i+1 runs while the sampling warps work on tile i.
// Every wait is bounded: a wait that runs out raises the block's abort flag,
// which every other wait sees; the roles then stop, the producer and the MMA
// issuer wait (bounded) for what they issued, and the block frees its tensor
// memory and counts the timeout.
template <typename T, int CPT, int KP, int RB>
__global__ void __launch_bounds__(448, 1)
fwd_proj_ws_kernel(const __grid_constant__ CUtensorMap tmap,
                   const __grid_constant__ CUtensorMap fmap,
                   const __grid_constant__ CUtensorMap wmap, const KParams kp, const TileGeom tg,
                   const ProjGeom pg, int total, const T* __restrict__ input,
                   const T* __restrict__ bias, T* __restrict__ output, T* __restrict__ om_out) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int KB = pg.KB, NB = pg.NB, S = pg.S, sw = pg.sample_warps;
  const int npx = kp.tile_w * kp.tile_h;
  unsigned char* wsm = smem;                 // KB x NB x 128 B
  unsigned char* as = smem + pg.a_off;       // S x KB x 16 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pg.bar_off);
  uint64_t* wfull = bars;            // 1
  uint64_t* afull = bars + 1;        // 2 (S used)
  uint64_t* aempty = bars + 3;       // 2
  uint64_t* winfull = bars + 5;      // 2
  uint64_t* winempty = bars + 7;     // 2
  uint64_t* accfull = bars + 9;      // 2
  uint64_t* accempty = bars + 11;    // 2
  uint64_t* rowsfull = bars + 13;    // 2
  uint64_t* rowsempty = bars + 15;   // 2
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = kp.tiles_w * kp.tiles_h;
  const int gb = blockIdx.x % tg.ngb;  // the same for all of this block's tiles

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(pg.ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    mbar_init(wfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 1);
      mbar_init(&winfull[b], 1);
      mbar_init(&winempty[b], sw);
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
      mbar_init(&rowsfull[b], 4);
      mbar_init(&rowsempty[b], sw);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;

  auto tile_of = [&](int t, int& n, int& ho0, int& wo0) {
    const int rest = t / tg.ngb;
    const int tt = rest % tiles;
    n = rest / tiles;
    const int ty = tt / kp.tiles_w;
    ho0 = ty * kp.tile_h;
    wo0 = (tt - ty * kp.tiles_w) * kp.tile_w;
  };

  if (warp < sw) {
    // ---- sampling
    int i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const int b = i & 1;
      const uint32_t ph = (uint32_t)((i >> 1) & 1);
      if (!wait_or_abort(&rowsfull[b], ph, abort)) break;
      if (!wait_or_abort(&winfull[b], ph, abort)) break;
      int n, ho0, wo0;
      tile_of(t, n, ho0, wo0);
      const int wy0 = ho0 * kp.stride_h + tg.org_y, wx0 = wo0 * kp.stride_w + tg.org_x;
      const T* oms = reinterpret_cast<const T*>(smem + pg.rows_off + b * pg.rows_stride);
      const unsigned char* win = smem + pg.win_off + b * pg.win_stride;
      sample_tile<T, CPT, KP, RB>(kp, tg, pg, threadIdx.x, n, gb, ho0, wo0, wy0, wx0, oms, win,
                                  true, input, output);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&rowsempty[b]);
        mbar_arrive(&winempty[b]);
      }
    }
  } else if (warp == sw && lane == 0) {
    // ---- producer
    mbar_expect_tx(wfull, (uint32_t)(KB * NB * 128));
    for (int kb = 0; kb < KB; ++kb)
      tma_load_2d(wsm + kb * NB * 128, &wmap, wfull, kb * 64, gb * NB);
    int i = 0, last_a = -1, last_w = -1;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const int b = i & 1, st = i % S;
      int n, ho0, wo0;
      tile_of(t, n, ho0, wo0);
      const int wy0 = ho0 * kp.stride_h + tg.org_y, wx0 = wo0 * kp.stride_w + tg.org_x;
      if (!wait_or_abort(&aempty[st], (uint32_t)(((i / S) & 1) ^ 1), abort)) break;
      mbar_expect_tx(&afull[st], (uint32_t)(KB * npx * 128));
      for (int kb = 0; kb < KB; ++kb)
        tma_load_4d(as + (st * KB + kb) * 128 * 128, &fmap, &afull[st], kb * 64, wo0, ho0, n);
      last_a = i;
      if (!wait_or_abort(&winempty[b], (uint32_t)(((i >> 1) & 1) ^ 1), abort)) break;
      mbar_expect_tx(&winfull[b], tg.win_bytes);
      tma_load_4d(smem + pg.win_off + b * pg.win_stride, &tmap, &winfull[b],
                  gb * tg.GB * kp.gc, wx0, wy0, n);
      last_w = i;
    }
    if (*abort) {
      // no copy may still write this block's memory when it frees it: the
      // weights, and the latest copy into each buffer (bounded waits)
      mbar_wait_bounded(wfull, 0, kProjWaitPolls);
      for (int j = last_a - S + 1 > 0 ? last_a - S + 1 : 0; j <= last_a; ++j)
        mbar_wait_bounded(&afull[j % S], (uint32_t)((j / S) & 1), kProjWaitPolls);
      for (int j = last_w - 1 > 0 ? last_w - 1 : 0; j <= last_w; ++j)
        mbar_wait_bounded(&winfull[j & 1], (uint32_t)((j >> 1) & 1), kProjWaitPolls);
    }
  } else if (warp == sw + 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc =
        mma_idesc(std::is_same<T, __half>::value ? 0u : 1u, (uint32_t)NB, 128u);
    int last = -1;
    if (wait_or_abort(wfull, 0, abort)) {
      int i = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
        const int b = i & 1, st = i % S;
        if (!wait_or_abort(&afull[st], (uint32_t)((i / S) & 1), abort)) break;
        if (!wait_or_abort(&accempty[b], (uint32_t)(((i >> 1) & 1) ^ 1), abort)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(b * NB);
        for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sw128_desc(smem_addr(as + (st * KB + kb) * 128 * 128) + 32u * kk);
            const uint64_t bd = sw128_desc(smem_addr(wsm + kb * NB * 128) + 32u * kk);
            const uint32_t accum = (kb | kk) != 0;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
                : "memory");
          }
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&aempty[st]))
            : "memory");
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&accfull[b]))
            : "memory");
        last = i;
      }
    }
    // the MMAs already issued finish before tensor memory is freed
    if (*abort && last >= 0)
      mbar_wait_bounded(&accfull[last & 1], (uint32_t)((last >> 1) & 1), kProjWaitPolls);
  } else if (warp >= sw + 2 && warp < sw + 6) {
    // ---- rows: this warp's lane quarter of the accumulator
    const int q = warp & 3, r = q * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const int b = i & 1;
      const uint32_t ph = (uint32_t)((i >> 1) & 1);
      if (!wait_or_abort(&accfull[b], ph, abort)) break;
      if (!wait_or_abort(&rowsempty[b], ph ^ 1u, abort)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int n, ho0, wo0;
      tile_of(t, n, ho0, wo0);
      const int ho = ho0 + r / kp.tile_w, wo = wo0 + r % kp.tile_w;
      T* og = nullptr;
      if (om_out && r < npx && ho < kp.Ho && wo < kp.Wo)
        og = om_out + (((size_t)n * kp.Ho + ho) * kp.Wo + wo) * ((size_t)kp.G * pg.rs) + gb * NB;
      T* os = reinterpret_cast<T*>(smem + pg.rows_off + b * pg.rows_stride) + r * pg.om_stride;
      const uint32_t tb = tmem + (uint32_t)(b * NB) + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < NB; c += 16) {
        float v[16];
        tmem_ld16(tb + (uint32_t)c, v);  // every lane of the warp takes part
        if (r >= npx) continue;
        if (bias) {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] += Dt<T>::to_f(bias[gb * NB + c + e]);
        }
        uint32_t wv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) wv[e] = Dt<T>::pack(v + 2 * e);
        const uint4 lo = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        const uint4 hi = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        if (DCN_IN_SPAN(os + c, 32, smem + pg.rows_off + b * pg.rows_stride, pg.om_bytes,
                        kBadShared)) {
          reinterpret_cast<uint4*>(os + c)[0] = lo;
          reinterpret_cast<uint4*>(os + c)[1] = hi;
        }
        if (og) {
          reinterpret_cast<uint4*>(og + c)[0] = lo;
          reinterpret_cast<uint4*>(og + c)[1] = hi;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&accempty[b]);
        mbar_arrive(&rowsfull[b]);
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && *abort) atomicAdd(&g_proj_wait_timeouts, 1ull);
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(pg.ncols)
                 : "memory");
  }
}

template <typename T, int CPT>
cudaError_t launch_t(const CUtensorMap& map, const CUtensorMap& fmap, const CUtensorMap& wmap,
                     const KParams& kp, const TileGeom& tg, const ProjGeom& pg, const T* in,
                     const T* bias, T* out, T* om, cudaStream_t s) {
  constexpr int bytes = CPT * (int)sizeof(T);
  if constexpr (bytes >= 16 && bytes <= 64) {
    const bool r128 = (size_t)tg.GB * kp.gc * sizeof(T) == 128;
    auto k = kp.P == 9 ? (r128 ? fwd_proj_kernel<T, CPT, 9, 128> : fwd_proj_kernel<T, CPT, 9, 0>)
           : kp.P == 8 ? (r128 ? fwd_proj_kernel<T, CPT, 8, 128> : fwd_proj_kernel<T, CPT, 8, 0>)
                       : (r128 ? fwd_proj_kernel<T, CPT, 0, 128> : fwd_proj_kernel<T, CPT, 0, 0>);
    const long long grid = (long long)kp.N * kp.tiles_w * kp.tiles_h * tg.ngb;
    if (grid > INT_MAX / 2) return cudaErrorInvalidConfiguration;
    if (pg.ws) {
      auto kw = kp.P == 9 ? (r128 ? fwd_proj_ws_kernel<T, CPT, 9, 128> : fwd_proj_ws_kernel<T, CPT, 9, 0>)
              : kp.P == 8 ? (r128 ? fwd_proj_ws_kernel<T, CPT, 8, 128> : fwd_proj_ws_kernel<T, CPT, 8, 0>)
                          : (r128 ? fwd_proj_ws_kernel<T, CPT, 0, 128> : fwd_proj_ws_kernel<T, CPT, 0, 0>);
      cudaError_t e =
          cudaFuncSetAttribute(kw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pg.smem_bytes);
      if (e != cudaSuccess) return e;
      int dev = 0, sms = 0;
      if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
      // one block per SM, a multiple of the group-block count: each block then
      // projects one group block's rows throughout
      long long blocks = sms / tg.ngb * tg.ngb;
      if (blocks < tg.ngb) blocks = tg.ngb;
      if (blocks > grid) blocks = grid;
      const int threads = (pg.sample_warps + 6) * 32;
      kw<<<(unsigned)blocks, threads, pg.smem_bytes, s>>>(map, fmap, wmap, kp, tg, pg, (int)grid, in,
                                                          bias, out, om);
      return cudaGetLastError();
    }
    cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pg.smem_bytes);
    if (e != cudaSuccess) return e;
    const int threads = (kp.tile_w * kp.tile_h * tg.GB * (kp.gc / CPT) + 31) / 32 * 32;
    if (threads > 256 || threads < 32 * ((kp.tile_w * kp.tile_h + 31) / 32))
      return cudaErrorInvalidConfiguration;
    k<<<(unsigned)grid, threads, pg.smem_bytes, s>>>(map, fmap, wmap, kp, tg, pg, in, bias, out,
                                                     om);
    return cudaGetLastError();
  } else {
    return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_d(const void* map, const void* fmap, const void* wmap, const KParams& kp,
                     const TileGeom& tg, const ProjGeom& pg, int cpt, const void* in,
                     const void* bias, void* out, void* om, cudaStream_t s) {
  const CUtensorMap& m = *static_cast<const CUtensorMap*>(map);
  const CUtensorMap& fm = *static_cast<const CUtensorMap*>(fmap);
  const CUtensorMap& wm = *static_cast<const CUtensorMap*>(wmap);
  const T* i_ = static_cast<const T*>(in);
  const T* b_ = static_cast<const T*>(bias);
  T* y_ = static_cast<T*>(out);
  T* o_ = static_cast<T*>(om);
  switch (cpt) {
    case 8: return launch_t<T, 8>(m, fm, wm, kp, tg, pg, i_, b_, y_, o_, s);
    case 16: return launch_t<T, 16>(m, fm, wm, kp, tg, pg, i_, b_, y_, o_, s);
    case 32: return launch_t<T, 32>(m, fm, wm, kp, tg, pg, i_, b_, y_, o_, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool proj_plan(const KParams& kp, const TileGeom& tg, int es, int K, int rs, ProjGeom* pg) {
  const int npx = kp.tile_w * kp.tile_h;
  const int NB = tg.GB * rs;
  if (npx > 128 || NB > 256 || NB % 16 || K % 64 || K > 256 || es != 2) return false;
  pg->ws = 0;
  pg->S = 1;
  pg->sample_warps = 0;
  pg->a_off = pg->rows_off = pg->win_stride = pg->rows_stride = 0;
  pg->KB = K / 64;
  pg->rs = rs;
  pg->NB = NB;
  pg->ncols = NB <= 32 ? 32 : NB <= 64 ? 64 : NB <= 128 ? 128 : 256;
  pg->om_stride = NB + 8;  // 16 bytes of padding: rows start in different banks
  pg->b_off = (unsigned)(pg->KB * 128 * 128);
  const unsigned opnd = (unsigned)(pg->KB * (128 + NB) * 128);
  pg->om_bytes = (unsigned)(npx * pg->om_stride * es);
  const unsigned region = opnd > pg->om_bytes ? opnd : pg->om_bytes;
  pg->win_off = (region + 1023u) & ~1023u;
  pg->bar_off = (pg->win_off + tg.win_bytes + 15u) & ~15u;
  pg->smem_bytes = pg->bar_off + 64u + 1024u;  // barriers and tensor-memory slot, alignment slack
  return pg->smem_bytes <= 227u * 1024u;
}

bool proj_plan_ws(const KParams& kp, const TileGeom& tg, int es, int K, int rs, int cpt,
                  ProjGeom* pg) {
  const int npx = kp.tile_w * kp.tile_h;
  const int NB = tg.GB * rs;
  const int sample_threads = npx * tg.GB * (kp.gc / cpt);
  if (npx > 128 || NB > 256 || NB % 16 || K % 64 || K > 256 || es != 2 || sample_threads > 256)
    return false;
  auto up = [](unsigned v, unsigned a) { return (v + a - 1) / a * a; };
  pg->ws = 1;
  pg->KB = K / 64;
  pg->rs = rs;
  pg->NB = NB;
  pg->ncols = 2 * NB <= 32 ? 32 : 2 * NB <= 64 ? 64 : 2 * NB <= 128 ? 128 : 2 * NB <= 256 ? 256 : 512;
  pg->om_stride = NB + 8;
  pg->sample_warps = (sample_threads + 31) / 32;
  pg->om_bytes = (unsigned)(npx * pg->om_stride * es);
  const unsigned wbytes = (unsigned)(pg->KB * NB * 128), abytes = (unsigned)(pg->KB * 128 * 128);
  const unsigned win = up(tg.win_bytes, 1024u), rows = up(pg->om_bytes, 16u);
  for (int S = 2; S >= 1; --S) {
    pg->S = S;
    pg->b_off = 0;
    pg->a_off = up(wbytes, 1024u);
    pg->win_off = up(pg->a_off + S * abytes, 1024u);
    pg->win_stride = win;
    pg->rows_off = pg->win_off + 2 * win;
    pg->rows_stride = rows;
    pg->bar_off = up(pg->rows_off + 2 * rows, 16u);
    pg->smem_bytes = pg->bar_off + 256u + 1024u;
    if (pg->smem_bytes <= 227u * 1024u) return true;
  }
  return false;
}

// The window budget the persistent kernel leaves for each of its two windows
// once the weights, the feature stages and the row buffers are placed (at
// most 64 KB; 0 if they do not fit).
size_t proj_ws_window_budget(const KParams& kp, const TileGeom& tg, int es, int K, int rs) {
  const size_t npx = (size_t)kp.tile_w * kp.tile_h, NB = (size_t)tg.GB * rs, KB = K / 64;
  const size_t fixed = KB * NB * 128 + 2 * KB * 128 * 128 + 2 * ((npx * (NB + 8) * es + 15) / 16 * 16) +
                      4096;
  const size_t cap = 227 * 1024;
  if (fixed >= cap) return 0;
  const size_t per = (cap - fixed) / 2 / 1024 * 1024;
  return per < 64 * 1024 ? per : 64 * 1024;
}

bool encode_proj_maps(const KParams& kp, const ProjGeom& pg, int dtype, const void* feat, int K,
                      const void* w, void* fmap_out, void* wmap_out) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc || (dtype != DCN_F16 && dtype != DCN_BF16)) return false;
  const CUtensorMapDataType dt =
      dtype == DCN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t es = 2;
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  // the features (K, Wo, Ho, N): a tile's pixels, 64 channels per copy
  const cuuint64_t fd[4] = {(cuuint64_t)K, (cuuint64_t)kp.Wo, (cuuint64_t)kp.Ho,
                            (cuuint64_t)kp.N};
  const cuuint64_t fs[3] = {(cuuint64_t)K * es, (cuuint64_t)kp.Wo * K * es,
                            (cuuint64_t)kp.Ho * kp.Wo * K * es};
  const cuuint32_t fb[4] = {64u, (cuuint32_t)kp.tile_w, (cuuint32_t)kp.tile_h, 1u};
  if (enc(static_cast<CUtensorMap*>(fmap_out), dt, 4, const_cast<void*>(feat), fd, fs, fb, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // the weight (K, G * row_stride): a block's NB rows, 64 channels per copy
  const cuuint64_t wd[2] = {(cuuint64_t)K, (cuuint64_t)kp.G * pg.rs};
  const cuuint64_t ws[1] = {(cuuint64_t)K * es};
  const cuuint32_t wb[2] = {64u, (cuuint32_t)pg.NB};
  return enc(static_cast<CUtensorMap*>(wmap_out), dt, 2, const_cast<void*>(w), wd, ws, wb, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t launch_fwd_proj(const void* map, const void* fmap, const void* wmap,
                            const KParams& kp, const TileGeom& tg, const ProjGeom& pg, int dtype,
                            int cpt, const void* in, const void* bias, void* out, void* om,
                            cudaStream_t s) {
  switch (dtype) {
    case DCN_F16: return launch_d<__half>(map, fmap, wmap, kp, tg, pg, cpt, in, bias, out, om, s);
    case DCN_BF16:
      return launch_d<__nv_bfloat16>(map, fmap, wmap, kp, tg, pg, cpt, in, bias, out, om, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t read_proj_wait_timeouts(unsigned long long* count) {
  return cudaMemcpyFromSymbol(count, g_proj_wait_timeouts, sizeof(unsigned long long));
}

DCN_BOUNDS_READER(fwd_proj)

}  // namespace dcn
