// dcn_fwd_tma.cu -- the forward with the input window staged in shared memory.
//
// The FlashInternImage page, section 2.2, describes the fused kernel as
// block-scheduled with the input tile staged in shared memory.  Here a block
// covers an 8x8-style tile of output pixels for GB groups, and one tensor copy
// (TMA, cp.async.bulk.tensor) brings the input window those pixels can sample
// -- the footprint of their taps plus a halo of R pixels for the offsets --
// into shared memory while the threads load their offsets and masks.  Pixels
// of the window outside the image arrive as zeros, which is exactly the zero
// padding of the op, so a sample whose bilinear cell lies in the window reads
// its four corners from shared memory with no bounds logic.  A sample whose
// cell leaves the window (large offsets, rare) reads its corners from global
// memory as the wide forward does.  Same arithmetic as the wide forward
// (dcn_fwd.cu): binary32 locations, mixed-precision FMAs into float32.
//
// The block's wait for the copy is bounded.  If it runs out, the block counts
// it (dcn_wait_timeouts) and computes every sample from global memory, which
// gives the same result; before it exits it waits once more, bounded, so that
// no copy into its shared memory is left in flight.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "dcn_common.cuh"
#include "dcn_kernels.h"

namespace dcn {

__device__ unsigned long long g_wait_timeouts = 0;

// Polls of the barrier before a block gives up on its copy (each poll blocks
// for a hardware-defined time, so this is seconds, far beyond any copy).
constexpr int kWaitPolls = 1 << 22;
// the epilogue projection's A tile: 128 rows of 128 bytes from the first
// 1024-byte boundary of the window
constexpr uint32_t kOutABytes = 16384u + 1024u;

// The inverse for the accumulator (CPT floats = NC chunks of 4 floats when a
// chunk holds 4 channels... of the storage type): channel chunk c is in slot
// (c - rot) mod NC.  Chunks here are 16 bytes of storage, i.e. 16/sizeof(T)
// channels.
template <int CPT, typename T>
__device__ __forceinline__ void unrotate_acc_t(float (&acc)[CPT], int rot) {
  constexpr int PER = 16 / (int)sizeof(T);  // channels per 16-byte chunk
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

// RB: the bytes of one window pixel (GB * gc * sizeof(T)) when known at compile
// time (128, the usual case), else 0.  M64: the offsets and masks are DCNv4's
// merged 64-byte rows (P = 9, 16-bit; kp.merged_rows64), read whole (a
// separate instance, so that the separate tensors' instance is unchanged).
// CFS: the centre feature scale applied before the store (an output the
// input's size, stride 1): out = core * (1 - s) + x_proj * s with s the gate of
// the unit's logit and x_proj the input at the output pixel, which lies in the
// window at the zero-offset centre tap (a gate of 1 passes x_proj exactly).
// OUT: the output projection y = out W^T + b in the epilogue (a block holds
// every channel of its tile's pixels, C = 64): the outputs, rounded to the
// storage type as they would be stored, become the rows of a 128-byte swizzled
// K-major tile over the spent window, one row per tile pixel; one thread
// issues the four K = 16 tcgen05.mma of the 128 x n_out x 64 product into
// tensor memory (W, n_out x 64, arrived by a tensor copy with the window), and
// warps 0-1 read their pixels' rows back, add the bias and store y (N, Ho, Wo,
// n_out).  output is not written then.
template <typename T, int CPT, int KP, int RB, bool M64 = false, bool CFS = false,
          bool OUT = false>
__global__ void __launch_bounds__(256)
fwd_tile_kernel(const __grid_constant__ CUtensorMap tmap, const KParams kp, const TileGeom tg,
                const T* __restrict__ input, const T* __restrict__ offset,
                const T* __restrict__ mask, T* __restrict__ output,
                const T* __restrict__ logits, const __grid_constant__ CUtensorMap wmap,
                const T* __restrict__ bias, T* __restrict__ yout, int n_out, int ncols) {
  constexpr int NW = CPT * (int)sizeof(T) / 4;  // 32-bit words per corner slice
  constexpr int NC = NW / 4;                    // 16-byte chunks per corner slice
  extern __shared__ __align__(128) unsigned char smem[];
  // the window's barrier; with OUT also the weight tile's, the MMAs', and the
  // tensor-memory address
  // with OUT the A tile (16 KB from the first 1024-byte boundary) lies over the
  // window, which is extended to hold it
  const uint32_t wend = OUT && tg.win_bytes < kOutABytes ? kOutABytes : tg.win_bytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + wend);
  uint64_t* wbar = bar + 1;
  uint64_t* mbar = bar + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 3);
  const int chunks = kp.gc / CPT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the swizzled operand tiles need 1024-byte aligned addresses: A over the
  // window, B (the weights) after the barriers
  const uint32_t sbase = smem_addr(smem);
  unsigned char* atile = smem + ((1024u - (sbase & 1023u)) & 1023u);
  unsigned char* btile = smem + wend + 64u + ((1024u - ((sbase + wend + 64u) & 1023u)) & 1023u);

  // block -> (image, tile, group block), the group block fastest: the blocks
  // of one tile copy neighbouring channels of the same window pixels
  const int gb = blockIdx.x % tg.ngb;
  const int rest = blockIdx.x / tg.ngb;
  const int tiles = kp.tiles_w * kp.tiles_h;
  const int t = rest % tiles, n = rest / tiles;
  const int ty = t / kp.tiles_w;
  const int ho0 = ty * kp.tile_h, wo0 = (t - ty * kp.tiles_w) * kp.tile_w;
  const int wy0 = ho0 * kp.stride_h + tg.org_y, wx0 = wo0 * kp.stride_w + tg.org_x;

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    if constexpr (OUT) {
      mbar_init(wbar, 1);
      mbar_init(mbar, 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, tg.win_bytes);
    tma_load_4d(smem, &tmap, bar, gb * tg.GB * kp.gc, wx0, wy0, n);
    if constexpr (OUT) {
      mbar_expect_tx(wbar, (uint32_t)n_out * 128u);
      tma_load_2d(btile, &wmap, wbar, 0, 0);
    }
  }
  // with OUT, once the copies are on their way: the bias as float32 after the
  // weight tile, and the tensor memory (the accumulator's n_out columns,
  // ncols a power of two), whose address the epilogue reads after a barrier
  float* sbias = reinterpret_cast<float*>(btile + n_out * 128);
  if constexpr (OUT) {
    for (int i = threadIdx.x; i < n_out; i += blockDim.x)
      sbias[i] = bias ? Dt<T>::to_f(bias[i]) : 0.f;
    __syncwarp();
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(tslot)),
                   "r"(ncols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
  }

  // thread -> (pixel of the tile, group of the block, channel slice)
  const int per_px = tg.GB * chunks;
  const int lp = threadIdx.x / per_px, r = threadIdx.x - lp * per_px;
  const int gl = r / chunks, slice = r - gl * chunks;
  const int g = gb * tg.GB + gl, c0 = slice * CPT;
  const int ho = ho0 + lp / kp.tile_w, wo = wo0 + lp % kp.tile_w;
  const bool active = lp < kp.tile_w * kp.tile_h && ho < kp.Ho && wo < kp.Wo;
  const uint32_t unit = active ? ((n * (uint32_t)kp.Ho + ho) * kp.Wo + wo) * kp.G + g : 0;

  const int P = KP > 0 ? KP : kp.P;
  const T* mrow = mask + (size_t)unit * kp.os_mask;
  const T* orow = offset + (size_t)unit * kp.os_off;
  if (!rows_in(kp, offset, mask, orow, mrow)) {  // (checked build) read unit 0's rows
    mrow = mask;
    orow = offset;
  }
  const T* img = input + (size_t)n * kp.H * kp.W * kp.C + g * kp.gc + c0;
  const uint32_t W = kp.W, H = kp.H, C = kp.C, WC = (uint32_t)kp.W * kp.C;
  const float ref_x = (float)(wo * kp.stride_w - kp.pad_w + kp.cen_w);
  const float ref_y = (float)(ho * kp.stride_h - kp.pad_h + kp.cen_h);
  const float scale = kp.offset_scale;

  UnitRows<T, KP> rows;
  bool vec = false;
  constexpr bool kVecRows = KP > 0 && (sizeof(T) == 2 || CPT <= 8);
  if constexpr (M64) {
    // DCNv4's merged 64-byte rows: the whole row in two 256-bit loads
    if (active && DCN_IN_SPAN(orow, 64, offset, offset_bytes<T>(kp), kBadRow)) {
      rows.load_merged64(orow);
      vec = true;
    }
  } else if constexpr (kVecRows) {
    vec = active && !kp.merged && rows.load(offset, mask, kp.units, orow, mrow);
  }

  float mx = 0.f, inv = 1.f;
  if (kp.softmax && active) {
    mx = -INFINITY;
    if (vec) {
#pragma unroll
      for (int p = 0; p < (KP > 0 ? KP : 1); ++p) mx = fmaxf(mx, rows.msk(p));
      float s = 0.f;
#pragma unroll
      for (int p = 0; p < (KP > 0 ? KP : 1); ++p) s += expf(rows.msk(p) - mx);
      inv = 1.f / s;
    } else {
      for (int p = 0; p < P; ++p) mx = fmaxf(mx, Dt<T>::one(mrow + p));
      float s = 0.f;
      for (int p = 0; p < P; ++p) s += expf(Dt<T>::one(mrow + p) - mx);
      inv = 1.f / s;
    }
  }

  const bool ready = mbar_wait_bounded(bar, 0, kWaitPolls);
  if (!ready && active && r == 0 && lp == 0) atomicAdd(&g_wait_timeouts, 1ull);

  float acc[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) acc[i] = 0.f;
  if (active) {
    // this thread's slice inside a window pixel, and the pixel's size
    const uint32_t rb = RB > 0 ? (uint32_t)RB : (uint32_t)(tg.GB * kp.gc) * (uint32_t)sizeof(T);
    const uint32_t wrb = (uint32_t)tg.WW * rb;  // one window row
    const uint32_t chunk0 = (uint32_t)(gl * kp.gc + c0) * (uint32_t)sizeof(T) / 16u;
    // A 16-byte shared load is served eight lanes at a time: the lanes of two
    // (or four) tile pixels.  Their window pixels are unrelated, so reading
    // the slices' chunks in the same order would hit the same banks; each
    // tile pixel slot starts its chunks at its own rotation instead, and the
    // accumulator is rotated back before the store.
    const int rot = NC > 1 ? lp & (NC - 1) : 0;
    uint32_t coff[NC];  // byte offset in a window pixel of accumulator chunk j
#pragma unroll
    for (int j = 0; j < NC; ++j) coff[j] = 16u * (chunk0 + (uint32_t)((j + rot) & (NC - 1)));
    const int WWm = tg.WW - 1, WHm = tg.WH - 1;

    // points whose cell leaves the window (rare) are marked here and done
    // after the loop, so that the unrolled loop holds only the shared-memory
    // path
    unsigned long long far = 0ull;
    // the point loop, compiled once with the rows in registers (V) and once
    // reading them from memory point by point
    auto points = [&](auto rows_in_regs) {
      constexpr bool V = decltype(rows_in_regs)::value;
#pragma unroll(KP > 0 ? KP : 1)
      for (int p = 0; p < P; ++p) {
        float m;
        float2 d;
        if constexpr (KP > 0 && V) {
          m = rows.msk(KP > 0 ? p : 0);
          d = rows.off(KP > 0 ? p : 0);
        } else {
          m = ld_once_1(mrow + p);
          d = ld_once_2(orow + 2 * p);
        }
        if (kp.softmax) m = expf(m - mx) * inv;
        const float x = location(d.x, kp.tap_x[p], scale, ref_x);
        const float y = location(d.y, kp.tap_y[p], scale, ref_y);
        if (!in_box(x, y, kp.W, kp.H)) continue;  // also NaN / inf
        const float xf = floorf(x), yf = floorf(y);
        const int cx = (int)xf - wx0, cy = (int)yf - wy0;
        if (!(ready && (unsigned)cx < (unsigned)WWm && (unsigned)cy < (unsigned)WHm)) {
          far |= 1ull << p;
          continue;
        }
        // the cell is in the window: corners from shared memory, zeros standing
        // for pixels outside the image
        const float fx = x - xf, fy = y - yf, gx = 1.f - fx, gy = 1.f - fy;
        const float gym = gy * m, fym = fy * m;
        const unsigned char* a00 = smem + (uint32_t)(cy * tg.WW + cx) * rb;
        const uint32_t at[4] = {0u, rb, wrb, wrb + rb};  // the corners' offsets
        const float w[4] = {gym * gx, gym * fx, fym * gx, fym * fx};
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t v[NW];
  #pragma unroll
          for (int j = 0; j < NC; ++j) {
            // accumulator chunk j takes the slice's chunk (j + rot) mod NC;
            // plain loads, so that the compiler may fold constant offsets
            const unsigned char* q = a00 + coff[j] + at[k];
            const uint4 c = DCN_IN_SPAN(q, 16, smem, tg.win_bytes, kBadShared)
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
    };
    if (KP > 0 && vec)
      points(std::true_type{});
    else
      points(std::false_type{});
    // far points: the point again, clamped corners from global memory,
    // weight 0 outside the image
    while (far) {
      const int p = __ffsll((long long)far) - 1;
      far &= far - 1;
      float m = ld_once_1(mrow + p);
      const float2 d = ld_once_2(orow + 2 * p);
      if (kp.softmax) m = expf(m - mx) * inv;
      const float x = location(d.x, kp.tap_x[p], scale, ref_x);
      const float y = location(d.y, kp.tap_y[p], scale, ref_y);
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
    unrotate_acc_t<CPT, T>(acc, rot);
    if constexpr (CFS) {
      // the gate of the unit's logit (logits (N, Ho, Wo, G): index = unit), and
      // x_proj = the input at (ho, wo), this thread's channels: from the window
      // (in natural chunk order), or from memory if the copy did not land
      const float sg = cfs_gate(DCN_IN_SPAN(logits + unit, sizeof(T), logits,
                                            (size_t)kp.units * sizeof(T), kBadRow)
                                    ? Dt<T>::one(logits + unit)
                                    : 0.f);
      const int cy = ho - wy0, cx = wo - wx0;
      uint32_t xw[NW];
      if (ready && (unsigned)cy < (unsigned)tg.WH && (unsigned)cx < (unsigned)tg.WW) {
        const unsigned char* q = smem + (uint32_t)(cy * tg.WW + cx) * rb + 16u * chunk0;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const uint4 c = DCN_IN_SPAN(q + 16 * j, 16, smem, tg.win_bytes, kBadShared)
                              ? *reinterpret_cast<const uint4*>(q + 16 * j)
                              : make_uint4(0u, 0u, 0u, 0u);
          xw[4 * j] = c.x;
          xw[4 * j + 1] = c.y;
          xw[4 * j + 2] = c.z;
          xw[4 * j + 3] = c.w;
        }
      } else {
        ldg_words_in<NW>(img + ((uint32_t)ho * WC + (uint32_t)wo * C), xw, input,
                         input_bytes<T>(kp));
      }
      float xv[CPT];
#pragma unroll
      for (int i = 0; i < NW; ++i) Dt<T>::unpack(xw[i], xv + i * Dt<T>::kPerWord);
#pragma unroll
      for (int i = 0; i < CPT; ++i) acc[i] = fmaf(sg, xv[i], (1.f - sg) * acc[i]);
    }
    if constexpr (!OUT) {
      if (out_in(kp, output, output + (size_t)unit * kp.gc + c0, CPT))
        Slice<T, CPT>::store(output + (size_t)unit * kp.gc + c0, acc);
    }
  }
  if constexpr (OUT) {
    // every thread is done with the window (which becomes the A tile), and
    // no copy into it is still in flight
    bool ok = ready || mbar_wait_bounded(bar, 0, kWaitPolls);
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;
    if (ok && active) {
      // the unit's outputs, rounded as stored, into row lp of the A tile:
      // channels gl*gc + c0 .. + CPT of the pixel, i.e. 16-byte chunks k0 ..
      // k0 + NC - 1 of its 128-byte row, each at position k ^ (row % 8)
      uint32_t wv[NW];
#pragma unroll
      for (int i = 0; i < NW; ++i) wv[i] = Dt<T>::pack(acc + i * Dt<T>::kPerWord);
      const uint32_t k0 = (uint32_t)(gl * kp.gc + c0) * (uint32_t)sizeof(T) / 16u;
      unsigned char* row = atile + (uint32_t)(lp >> 3) * 1024u + (uint32_t)(lp & 7) * 128u;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        unsigned char* q = row + 16u * ((k0 + (uint32_t)j) ^ (uint32_t)(lp & 7));
        if (DCN_IN_SPAN(q, 16, smem, wend, kBadShared))
          *reinterpret_cast<uint4*>(q) =
              make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
      }
    }
    // the A tile's writes to the tensor cores' view of shared memory
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    bool issued = false;
    if (threadIdx.x == 0 && ok) {
      ok = mbar_wait_bounded(wbar, 0, kWaitPolls);
      if (ok) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t idesc =
            mma_idesc(std::is_same<T, __half>::value ? 0u : 1u, (uint32_t)n_out, 128u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(smem_addr(atile) + 32u * kk);
          const uint64_t bd = sw128_desc(smem_addr(btile) + 32u * kk);
          const uint32_t accum = kk != 0;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(mbar))
            : "memory");
        issued = true;
        ok = mbar_wait_bounded(mbar, 0, kWaitPolls);  // the rest wait at the barrier
      }
    }
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!ok && threadIdx.x == 0) {
      atomicAdd(&g_wait_timeouts, 1ull);
      // nothing may still write this block's memory when it goes on
      mbar_wait_bounded(wbar, 0, kWaitPolls);
      if (issued) mbar_wait_bounded(mbar, 0, kWaitPolls);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // warp w reads tensor-memory lanes 32 (w % 4) .. + 31; the tile's pixels
    // are rows 0 .. npx - 1, so the warps of the first (npx + 31) / 32 lane
    // quarters share the columns: warp w takes 16-column chunks w / 4,
    // w / 4 + J, ... of its quarter's J warps, two chunks per wait
    const int npx = kp.tile_w * kp.tile_h;
    const int qw = warp & 3, nwarps = (int)(blockDim.x >> 5);
    if (ok && qw * 32 < npx) {
      const int J = (nwarps - qw + 3) >> 2, nch = n_out >> 4;
      const int px = qw * 32 + lane;
      const int ph = ho0 + px / kp.tile_w, pw = wo0 + px % kp.tile_w;
      const bool live = px < npx && ph < kp.Ho && pw < kp.Wo;
      T* dst = yout + (((size_t)n * kp.Ho + ph) * kp.Wo + pw) * (size_t)n_out;
      const uint32_t tb = tmem + ((uint32_t)(qw * 32) << 16);
      for (int ch = warp >> 2; ch < nch; ch += 2 * J) {
        const int ch2 = ch + J < nch ? ch + J : ch;  // the same chunk twice when alone
        uint32_t ra[16], rb[16];
        tmem_ld16x2(tb + (uint32_t)(ch * 16), tb + (uint32_t)(ch2 * 16), ra, rb);
        if (!live) continue;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (hh && ch2 == ch) break;
          const uint32_t* rr = hh ? rb : ra;
          const int c = (hh ? ch2 : ch) * 16;
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rr[i]) + sbias[c + i];
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = Dt<T>::pack(v + 2 * i);
          if (DCN_IN_SPAN(dst + c, 32, yout, (size_t)kp.N * kp.Ho * kp.Wo * n_out * sizeof(T),
                          kBadStore)) {
            reinterpret_cast<uint4*>(dst + c)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4*>(dst + c)[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();  // tensor memory is read
    if (warp == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(ncols)
                   : "memory");
    }
    return;
  }
  // a block whose wait ran out leaves no copy in flight into its memory
  if (!ready) mbar_wait_bounded(bar, 0, kWaitPolls);
}

// ---- host side ------------------------------------------------------------------

// The CUDA driver's tensor-map encoder, looked up once through the runtime (the
// library links the runtime only).
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

void* tensor_map_encoder() { return reinterpret_cast<void*>(encoder()); }

bool encode_input_map(const KParams& kp, const TileGeom& tg, int dtype, const void* input,
                      void* map_out) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  CUtensorMapDataType dt;
  size_t es;
  switch (dtype) {
    case DCN_F32: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; es = 4; break;
    case DCN_F16: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; es = 2; break;
    case DCN_BF16: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; es = 2; break;
    default: return false;
  }
  const cuuint64_t dims[4] = {(cuuint64_t)kp.C, (cuuint64_t)kp.W, (cuuint64_t)kp.H,
                              (cuuint64_t)kp.N};
  const cuuint64_t strides[3] = {(cuuint64_t)kp.C * es, (cuuint64_t)kp.W * kp.C * es,
                                 (cuuint64_t)kp.H * kp.W * kp.C * es};
  const cuuint32_t box[4] = {(cuuint32_t)(tg.GB * kp.gc), (cuuint32_t)tg.WW,
                             (cuuint32_t)tg.WH, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMap* m = static_cast<CUtensorMap*>(map_out);
  return enc(m, dt, 4, const_cast<void*>(input), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output projection of the epilogue (fwd_tile_kernel OUT): the weight's
// tensor map, the bias (or nullptr), the projection's output and its width.
struct OutProj {
  const CUtensorMap* wmap = nullptr;
  const void* bias = nullptr;
  void* y = nullptr;
  int n_out = 0;
};

template <typename T, int CPT, bool CFS>
static auto out_instance(int P) {
  return P == 9 ? fwd_tile_kernel<T, CPT, 9, 128, false, CFS, true>
       : P == 8 ? fwd_tile_kernel<T, CPT, 8, 128, false, CFS, true>
                : fwd_tile_kernel<T, CPT, 0, 128, false, CFS, true>;
}

template <typename T, int CPT>
static cudaError_t launch_tile_t(const CUtensorMap& map, const KParams& kp, const TileGeom& tg,
                                 const T* i_, const T* o_, const T* m_, T* y_, const T* l_,
                                 const OutProj& op, cudaStream_t s) {
  constexpr int bytes = CPT * (int)sizeof(T);
  if constexpr (bytes >= 16 && bytes <= 64) {
    const bool out = op.y != nullptr;
    // the window, then the barriers (and with the projection the weight tile,
    // 1024-byte aligned)
    const size_t smem = out ? (size_t)(tg.win_bytes < kOutABytes ? kOutABytes : tg.win_bytes) +
                                  64 + 1024 + (size_t)op.n_out * (128 + 4)
                            : tg.win_bytes + 16;
    int ncols = 32;
    while (ncols < op.n_out) ncols *= 2;
    const bool r128 = (size_t)tg.GB * kp.gc * sizeof(T) == 128;
    auto k = kp.P == 9 ? (r128 ? fwd_tile_kernel<T, CPT, 9, 128> : fwd_tile_kernel<T, CPT, 9, 0>)
           : kp.P == 8 ? (r128 ? fwd_tile_kernel<T, CPT, 8, 128> : fwd_tile_kernel<T, CPT, 8, 0>)
                       : (r128 ? fwd_tile_kernel<T, CPT, 0, 128> : fwd_tile_kernel<T, CPT, 0, 0>);
    if constexpr (sizeof(T) == 2) {
      if (kp.P == 9 && kp.merged && kp.merged_rows64)
        k = r128 ? fwd_tile_kernel<T, CPT, 9, 128, true> : fwd_tile_kernel<T, CPT, 9, 0, true>;
      // the centre feature scale in the epilogue (separate offset / mask tensors)
      if (l_)
        k = kp.P == 9 ? (r128 ? fwd_tile_kernel<T, CPT, 9, 128, false, true>
                              : fwd_tile_kernel<T, CPT, 9, 0, false, true>)
          : kp.P == 8 ? (r128 ? fwd_tile_kernel<T, CPT, 8, 128, false, true>
                              : fwd_tile_kernel<T, CPT, 8, 0, false, true>)
                      : (r128 ? fwd_tile_kernel<T, CPT, 0, 128, false, true>
                              : fwd_tile_kernel<T, CPT, 0, 0, false, true>);
      // the output projection in the epilogue: 64 channels (128-byte pixels)
      // of all groups in the block, at most 64 tile pixels
      if (out) {
        if constexpr (CPT == 8 || CPT == 16) {
          if (!r128 || tg.ngb != 1 || kp.merged || kp.tile_w * kp.tile_h > 64 ||
              op.n_out % 16 || op.n_out < 16 || op.n_out > 128)
            return cudaErrorInvalidValue;
          k = l_ ? out_instance<T, CPT, true>(kp.P) : out_instance<T, CPT, false>(kp.P);
        } else {
          return cudaErrorInvalidValue;
        }
      }
    } else {
      if (l_ || out) return cudaErrorInvalidValue;
    }
    if (smem > 48 * 1024) {
      cudaError_t e =
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    const long long grid = (long long)kp.N * kp.tiles_w * kp.tiles_h * tg.ngb;
    if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
    // one thread per (tile pixel, group of the block, channel slice), in whole
    // warps: 256 for the power-of-two tiles, fewer for tiles such as 7 x 7
    const int threads = (kp.tile_w * kp.tile_h * tg.GB * (kp.gc / CPT) + 31) / 32 * 32;
    if (threads > 256) return cudaErrorInvalidConfiguration;
    k<<<(unsigned)grid, threads, smem, s>>>(map, kp, tg, i_, o_, m_, y_, l_,
                                            out ? *op.wmap : map,
                                            static_cast<const T*>(op.bias),
                                            static_cast<T*>(op.y), op.n_out, ncols);
    return cudaGetLastError();
  } else {
    return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_tile_d(const CUtensorMap& map, const KParams& kp, const TileGeom& tg,
                                 int cpt, const void* in, const void* off, const void* msk,
                                 void* out, const void* logits, const OutProj& op,
                                 cudaStream_t s) {
  const T* i_ = static_cast<const T*>(in);
  const T* o_ = static_cast<const T*>(off);
  const T* m_ = static_cast<const T*>(msk);
  const T* l_ = static_cast<const T*>(logits);
  T* y_ = static_cast<T*>(out);
  switch (cpt) {
    case 4: return launch_tile_t<T, 4>(map, kp, tg, i_, o_, m_, y_, l_, op, s);
    case 8: return launch_tile_t<T, 8>(map, kp, tg, i_, o_, m_, y_, l_, op, s);
    case 16: return launch_tile_t<T, 16>(map, kp, tg, i_, o_, m_, y_, l_, op, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_tile(const void* map, const KParams& kp, const TileGeom& tg, int dtype,
                            int cpt, const void* in, const void* off, const void* msk, void* out,
                            cudaStream_t s, const void* logits, const void* wmap,
                            const void* bias, void* y, int n_out) {
  const CUtensorMap& m = *static_cast<const CUtensorMap*>(map);
  OutProj op;
  if (y) {
    op.wmap = static_cast<const CUtensorMap*>(wmap);
    op.bias = bias;
    op.y = y;
    op.n_out = n_out;
  }
  switch (dtype) {
    case DCN_F32: return launch_tile_d<float>(m, kp, tg, cpt, in, off, msk, out, logits, op, s);
    case DCN_F16: return launch_tile_d<__half>(m, kp, tg, cpt, in, off, msk, out, logits, op, s);
    case DCN_BF16:
      return launch_tile_d<__nv_bfloat16>(m, kp, tg, cpt, in, off, msk, out, logits, op, s);
    default: return cudaErrorInvalidValue;
  }
}

// The output projection's weight (n_out rows of 64 channels) as one
// 128-byte swizzled box, the B operand of the epilogue's MMAs.
bool encode_out_weight_map(int dtype, const void* w, int n_out, void* map_out) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc || (dtype != DCN_F16 && dtype != DCN_BF16)) return false;
  const CUtensorMapDataType dt =
      dtype == DCN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t dims[2] = {64u, (cuuint64_t)n_out};
  const cuuint64_t strides[1] = {64u * 2u};
  const cuuint32_t box[2] = {64u, (cuuint32_t)n_out};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(static_cast<CUtensorMap*>(map_out), dt, 2, const_cast<void*>(w), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t read_wait_timeouts(unsigned long long* count) {
  return cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned long long));
}

DCN_BOUNDS_READER(fwd_tma)

}  // namespace dcn
