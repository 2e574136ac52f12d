// dcn_api.cu -- the C ABI of libdcn_b300 (declared in include/dcn_core.h):
// argument validation, the choice of kernel instance, and the launches.
//
// Every check runs on the host before the first CUDA call, so a rejected
// call leaves the device untouched.  No entry point allocates memory.
#include <algorithm>
#include <initializer_list>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/dcn_core.h"
#include "dcn_kernels.h"
#include "dcn_options.h"

namespace {

int elem_size(int dtype) {
  switch (dtype) {
    case DCN_F32: return 4;
    case DCN_F16: return 2;
    case DCN_BF16: return 2;
    default: return 0;
  }
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Largest coordinate magnitude for which integer pixel positions stay exact
// in binary32 with room to spare.
constexpr long long kMaxExtent = 1LL << 22;

struct Geometry {
  int Ho, Wo, P;
  long long n_in, n_out, units;  // elements of input/output, (pixel, group) pairs
};

int validate(const dcn_params_t* p, Geometry* g) {
  if (!p) return DCN_ERR_NULL;
  if (elem_size(p->dtype) == 0) return DCN_ERR_DTYPE;
  if (p->N < 0 || p->H < 1 || p->W < 1 || p->G < 1 || p->gc < 1) return DCN_ERR_SHAPE;
  if (p->kernel_h < 1 || p->kernel_w < 1 || p->stride_h < 1 || p->stride_w < 1 ||
      p->dilation_h < 1 || p->dilation_w < 1 || p->pad_h < 0 || p->pad_w < 0)
    return DCN_ERR_SHAPE;
  if (p->remove_center != 0 && p->remove_center != 1) return DCN_ERR_SHAPE;
  if (p->softmax != 0 && p->softmax != 1) return DCN_ERR_SHAPE;
  if (p->remove_center && (p->kernel_h % 2 == 0 || p->kernel_w % 2 == 0)) return DCN_ERR_SHAPE;
  if (!std::isfinite(p->offset_scale)) return DCN_ERR_SHAPE;
  const long long kk = (long long)p->kernel_h * p->kernel_w;
  const long long P = kk - p->remove_center;
  if (P > DCN_MAX_POINTS) return DCN_ERR_UNSUPPORTED;
  const long long C = (long long)p->G * p->gc;
  if (C > DCN_MAX_CHANNELS) return DCN_ERR_UNSUPPORTED;
  const long long Hp = (long long)p->H + 2LL * p->pad_h, Wp = (long long)p->W + 2LL * p->pad_w;
  const long long eh = (long long)p->dilation_h * (p->kernel_h - 1) + 1;
  const long long ew = (long long)p->dilation_w * (p->kernel_w - 1) + 1;
  if (Hp > kMaxExtent || Wp > kMaxExtent || eh > kMaxExtent || ew > kMaxExtent)
    return DCN_ERR_UNSUPPORTED;
  if (Hp < eh || Wp < ew) return DCN_ERR_SHAPE;
  const long long Ho = (Hp - eh) / p->stride_h + 1, Wo = (Wp - ew) / p->stride_w + 1;
  g->Ho = (int)Ho;
  g->Wo = (int)Wo;
  g->P = (int)P;
  // element counts must fit comfortably in 62 bits
  const long long lim = 1LL << 62;
  const long long hw = (long long)p->H * p->W;
  if (p->N > 0 && (hw > lim / p->N / C || Ho * Wo > lim / p->N / C / (2 * P)))
    return DCN_ERR_UNSUPPORTED;
  g->n_in = (long long)p->N * hw * C;
  g->n_out = (long long)p->N * Ho * Wo * C;
  g->units = (long long)p->N * Ho * Wo * p->G;
  return DCN_OK;
}

dcn::FastDiv fast_div(uint32_t d) {
  // see dcn::FastDiv: s = ceil(log2 d), mul = floor(2^32 (2^s - d) / d) + 1
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  dcn::FastDiv f;
  f.mul = (uint32_t)(((1ull << 32) * ((1ull << s) - d)) / d + 1);
  f.shift = s;
  f.d = d;
  return f;
}

void fill_kparams(const dcn_params_t* p, const Geometry& g, dcn::KParams* kp) {
  std::memset(kp, 0, sizeof *kp);
  kp->N = p->N; kp->H = p->H; kp->W = p->W; kp->G = p->G; kp->gc = p->gc; kp->C = p->G * p->gc;
  kp->Ho = g.Ho; kp->Wo = g.Wo; kp->P = g.P;
  kp->stride_h = p->stride_h; kp->stride_w = p->stride_w;
  kp->pad_h = p->pad_h; kp->pad_w = p->pad_w;
  kp->cen_h = p->dilation_h * (p->kernel_h - 1) / 2;
  kp->cen_w = p->dilation_w * (p->kernel_w - 1) / 2;
  kp->offset_scale = p->offset_scale;
  kp->softmax = p->softmax;
  kp->units = g.units;
  kp->os_off = 2 * g.P;
  kp->os_mask = g.P;
  kp->merged = 0;
  kp->merged_rows64 = 0;
  kp->div_G = fast_div((uint32_t)p->G);
  kp->div_Wo = fast_div((uint32_t)g.Wo);
  kp->div_Ho = fast_div((uint32_t)g.Ho);
  // x-major point order: the kernel column outer, the row inner; the centre
  // tap deleted in place when asked.
  int k = 0;
  for (int ix = 0; ix < p->kernel_w; ++ix)
    for (int iy = 0; iy < p->kernel_h; ++iy) {
      if (p->remove_center && ix == (p->kernel_w - 1) / 2 && iy == (p->kernel_h - 1) / 2) continue;
      kp->tap_x[k] = (float)(ix * p->dilation_w - kp->cen_w);
      kp->tap_y[k] = (float)(iy * p->dilation_h - kp->cen_h);
      ++k;
    }
}

// Host-side fault hook for tests of the error path: with the fault_inject
// switch set, a valid call reports DCN_ERR_CUDA instead of launching.
bool fault_injected() { return dcn::options().fault_inject != 0; }

// Channels per thread of the forward.  The wide kernel (returned negated)
// takes slices of 16 channels (or 8, 4) of 16 to 64 bytes when the unit count
// and every image's element count fit in 31 bits and the input and output are
// 32-byte aligned (16 for a 16-byte slice).  Otherwise the general kernel with
// the widest power of two dividing gc up to one 16-byte vector (or
// the fwd_cpt switch), whose slices start aligned in both the input and the output.
int pick_fwd_cpt(const dcn_params_t* p, const Geometry& g, const void* in, const void* out) {
  const int es = elem_size(p->dtype);
  const long long img = (long long)p->H * p->W * p->G * p->gc;
  if (dcn::options().fwd_wide && img < (1LL << 31)) {
    const int wcap = dcn::options().fwd_wide_cpt;
    for (int c = 16; c >= 4; c >>= 1) {
      if (c > wcap) continue;
      const int bytes = c * es;
      if (p->gc % c || bytes < 16 || bytes > 64) continue;
      if (g.units * (p->gc / c) >= (1LL << 31)) continue;
      const size_t a = bytes >= 32 ? 32 : 16;
      if (aligned(in, a) && aligned(out, a)) return -c;
    }
  }
  int cap = (dcn::options().fwd_cpt > 0 ? dcn::options().fwd_cpt : 16 / es);
  for (int c = 32; c >= 1; c >>= 1) {
    if (c > cap || p->gc % c) continue;
    const size_t a = (size_t)(c * es < 16 ? c * es : 16);
    if (aligned(in, a) && aligned(out, a)) return c;
  }
  return 1;
}

// 2-D tiles for the wide forward: a block of 256 threads covers
// px = 256 / (G * gc/cpt) output pixels.  Of the power-of-two shapes tw x th
// = px, the one that pads the output plane least (then the squarest) is
// taken, and only when the padding wastes at most 20 % of the threads;
// otherwise (and when G times the slices per unit is not a power of two up to
// 256, or with the fwd_tile switch off) blocks take consecutive items.  Measured on
// B300: FlashInternImage-T stage 1 (56^2, 8x8 tiles) 79.9 -> 73.7 us,
// 64 x 28^2 x 128 fp32 131 -> 117 us, from better L1 reuse of the input;
// shapes that padded 7x7 or 13x13 planes by a third were slower.
void plan_fwd_tiles(const dcn_params_t* p, const Geometry& g, int cpt, dcn::KParams* kp) {
  kp->tile_w = kp->tile_h = kp->tiles_w = kp->tiles_h = 0;
  if (!dcn::options().fwd_tile) return;
  const long long per_px = (long long)p->G * (p->gc / cpt);
  if (per_px > 256 || (per_px & (per_px - 1))) return;
  const int px = (int)(256 / per_px);
  long long best = -1;
  int bw = 0, bh = 0;
  for (int tw = 1; tw <= px; tw <<= 1) {
    const int th = px / tw;
    const long long padded = (long long)((g.Wo + tw - 1) / tw) * tw * ((g.Ho + th - 1) / th) * th;
    const int skew = tw > th ? tw / th : th / tw;
    const int bskew = bw > bh ? (bh ? bw / bh : 0) : (bw ? bh / bw : 0);
    if (best < 0 || padded < best || (padded == best && skew < bskew)) {
      best = padded;
      bw = tw;
      bh = th;
    }
  }
  if (best * 5 > (long long)g.Wo * g.Ho * 6) return;  // more than 20 % padding
  const long long tiles_w = (g.Wo + bw - 1) / bw, tiles_h = (g.Ho + bh - 1) / bh;
  if ((long long)p->N * tiles_w * tiles_h > INT_MAX) return;
  kp->tile_w = bw;
  kp->tile_h = bh;
  kp->tiles_w = (int)tiles_w;
  kp->tiles_h = (int)tiles_h;
}

// The TMA-staged forward: the wide forward's slices, GB groups per block
// (all of them when a pixel's channels fit in 128 bytes, else the largest
// divisor of G that does), a power-of-two tile of 256 / (GB * gc/cpt) output
// pixels, and a window of the tile's footprint plus a halo of R pixels, R from
// 6 (the fwd_halo switch) down to 0 so that the window stays within kTileSmem (three
// blocks per SM).  Needs the input 16-byte aligned and every tensor-map
// stride a multiple of 16 bytes; fills the tensor map.  The fwd_tma switch at 0 turns it
// off.
constexpr size_t kTileSmem = 64 * 1024;

bool plan_fwd_tile(const dcn_params_t* p, const Geometry& g, int cpt, const void* in,
                   dcn::KParams* kp, dcn::TileGeom* tg, void* map, size_t budget = kTileSmem,
                   bool any_shape = false, int* halo = nullptr) {
  if (!dcn::options().fwd_tma) return false;
  const int es = elem_size(p->dtype);
  const long long C = (long long)p->G * p->gc;
  if (!aligned(in, 16) || (C * es) % 16 || (p->gc * es) % 16) return false;
  if ((long long)p->N * p->H * p->W * C >= (1LL << 40)) return false;
  int GB = 0;
  for (int d = p->G; d >= 1; --d)
    if (p->G % d == 0 && (long long)d * p->gc * es <= 128) {
      GB = d;
      break;
    }
  if (!GB) return false;
  const int chunks = p->gc / cpt;
  const int per_px = GB * chunks;
  if (per_px > 256 || (per_px & (per_px - 1))) return false;
  const int px = 256 / per_px;
  long long best = -1;
  int bw = 0, bh = 0;
  if (any_shape) {
    // any tw x th tile whose block (tw * th * per_px threads, rounded up to
    // whole warps) fits 256 threads: the fewest warps launched over the plane,
    // then the fewest blocks, then the squarest.  Small planes (14 x 14, 7 x 7)
    // take tiles such as 7 x 7 that no power-of-two shape matches.
    long long bblocks = 0;
    for (int tw = 1; tw <= px && tw <= g.Wo; ++tw)
      for (int th = 1; tw * th <= px && th <= g.Ho; ++th) {
        const long long blocks = (long long)((g.Wo + tw - 1) / tw) * ((g.Ho + th - 1) / th);
        const long long warps = blocks * ((tw * th * per_px + 31) / 32);
        const int skew = tw > th ? tw - th : th - tw, bskew = bw > bh ? bw - bh : bh - bw;
        if (best < 0 || warps < best || (warps == best && blocks < bblocks) ||
            (warps == best && blocks == bblocks && skew < bskew)) {
          best = warps;
          bblocks = blocks;
          bw = tw;
          bh = th;
        }
      }
    // more than 20 % of the launched lanes idle
    if (best * 32 * 5 > (long long)g.Wo * g.Ho * per_px * 6) return false;
  } else {
    // least-padding power-of-two tile of 256 threads, then the squarest
    for (int tw = 1; tw <= px; tw <<= 1) {
      const int th = px / tw;
      const long long padded = (long long)((g.Wo + tw - 1) / tw) * tw * ((g.Ho + th - 1) / th) * th;
      const int skew = tw > th ? tw / th : th / tw;
      const int bskew = bw > bh ? (bh ? bw / bh : 0) : (bw ? bh / bw : 0);
      if (best < 0 || padded < best || (padded == best && skew < bskew)) {
        best = padded;
        bw = tw;
        bh = th;
      }
    }
    if (best * 5 > (long long)g.Wo * g.Ho * 6) return false;  // more than 20 % padding
  }
  const double os = p->offset_scale;
  const int cw = p->dilation_w * (p->kernel_w - 1) / 2, ch = p->dilation_h * (p->kernel_h - 1) / 2;
  const double x0 = -cw * os, x1 = ((p->kernel_w - 1) * p->dilation_w - cw) * os;
  const double y0 = -ch * os, y1 = ((p->kernel_h - 1) * p->dilation_h - ch) * os;
  const int tmin_x = (int)std::floor(x0 < x1 ? x0 : x1), tmax_x = (int)std::ceil(x0 < x1 ? x1 : x0);
  const int tmin_y = (int)std::floor(y0 < y1 ? y0 : y1), tmax_y = (int)std::ceil(y0 < y1 ? y1 : y0);
  const size_t rb = (size_t)GB * p->gc * es;
  for (int R = dcn::options().fwd_halo; R >= 0; --R) {
    const long long WH = (long long)(bh - 1) * p->stride_h + (tmax_y - tmin_y) + 2 + 2 * R;
    const long long WW = (long long)(bw - 1) * p->stride_w + (tmax_x - tmin_x) + 2 + 2 * R;
    if (WH > 256 || WW > 256 || (size_t)(WH * WW) * rb > budget) continue;
    tg->GB = GB;
    tg->ngb = p->G / GB;
    tg->WH = (int)WH;
    tg->WW = (int)WW;
    tg->org_y = -p->pad_h + ch + tmin_y - R;
    tg->org_x = -p->pad_w + cw + tmin_x - R;
    tg->win_bytes = (unsigned)(WH * WW * rb);
    const long long tiles_w = (g.Wo + bw - 1) / bw, tiles_h = (g.Ho + bh - 1) / bh;
    if ((long long)p->N * tiles_w * tiles_h * tg->ngb > INT_MAX) return false;
    kp->tile_w = bw;
    kp->tile_h = bh;
    kp->tiles_w = (int)tiles_w;
    kp->tiles_h = (int)tiles_h;
    if (halo) *halo = R;
    return dcn::encode_input_map(*kp, *tg, p->dtype, in, map);
  }
  return false;
}

// Channels per thread of the backward: a power of two dividing gc, at most 4
// (or the bwd_cpt switch), with gc/c a power of two no larger than 32 so that a
// unit's threads are adjacent lanes of one warp; 0 selects the kernel that
// takes any gc.  Four float32 channels per lane make the lanes of one unit
// cover whole 32-byte sectors of grad_input in a single vector reduction,
// which halves the L2 reduction requests against one lane per 16 channels.
int pick_bwd_cpt(const dcn_params_t* p, const void* in, const void* gout, const void* acc) {
  const int es = elem_size(p->dtype);
  int cap = dcn::options().bwd_cpt;
  for (int c = 32; c >= 1; c >>= 1) {
    if (c > cap || p->gc % c) continue;
    const int chunks = p->gc / c;
    if (chunks > 32 || (chunks & (chunks - 1))) continue;
    const size_t a = (size_t)(c * es < 16 ? c * es : 16);
    const size_t af = c % 4 == 0 ? 16 : (c % 2 == 0 ? 8 : 4);
    if (aligned(in, a) && aligned(gout, a) && aligned(acc, af)) return c;
  }
  return 0;
}

// The split backward: a sample kernel shaped like the wide forward (same
// channels per thread and tiles, chosen here into *kp) and an input kernel
// over windows, one thread per output pixel of a TH x TW <= 256 tile of one
// (image, group).  Of the tile shapes, the one with the least work (tiles x
// (256 threads + window pixels)) is taken; the window is the tile's footprint
// plus a halo of R pixels for the offsets, R from 5 (the bwd_halo switch) down to 1
// so that the shared memory stays within kSplitSmem (four CTAs per SM).
// Needs gc*es of 16, 32 or 64 bytes, P <= 16, grad_out 32-byte aligned (16 for
// 16-byte rows) and the float32 accumulator 16-byte aligned.  Returns the
// sample kernel's channels per thread with *wg, *la, *lb filled, or 0.
//
// Used by default for 16-bit storage, where it measured fastest on B300
// (FlashInternImage-T stage 1, fp16: 308 us against 436 us for the
// single-pass kernel; InternImage-G stage 1, bf16: 391 us against 539 us for
// a fused window kernel since removed).  For float32 the corner gathers of
// the sample kernel cost twice as much and the single-pass kernel wins
// (64 x 28^2 x 128: 348 us against 227 us).  The bwd_split switch at 1 uses it
// for every dtype it can take, 0 never.
constexpr size_t kSplitSmem = 56 * 1024;
constexpr size_t kStageSmem = 32 * 1024;

int plan_split(const dcn_params_t* p, const Geometry& g, const void* in, const void* gout,
               const void* acc, dcn::KParams* kp, dcn::WinGeom* wg, int* la, int* lb) {
  const int mode = dcn::options().bwd_split;
  if (mode == 0 || (mode != 1 && p->dtype == DCN_F32)) return 0;
  const int es = elem_size(p->dtype);
  const int row = p->gc * es;
  if ((row != 16 && row != 32 && row != 64) || g.P > 16 || !aligned(acc, 16)) return 0;
  if ((long long)p->H * p->W >= (1LL << 31)) return 0;  // pixel offsets in 32 bits
  if (!aligned(gout, row >= 32 ? 32 : 16)) return 0;
  // the sample kernel: the wide forward's conditions, on input and grad_out
  const int cpt = -pick_fwd_cpt(p, g, in, gout);
  if (cpt <= 0) return 0;
  const int chunks = p->gc / cpt;
  if (chunks > 32 || (chunks & (chunks - 1))) return 0;
  // the input kernel's tile and window
  const double os = p->offset_scale;
  const int cw = p->dilation_w * (p->kernel_w - 1) / 2, ch = p->dilation_h * (p->kernel_h - 1) / 2;
  const double x0 = -cw * os, x1 = ((p->kernel_w - 1) * p->dilation_w - cw) * os;
  const double y0 = -ch * os, y1 = ((p->kernel_h - 1) * p->dilation_h - ch) * os;
  const int tmin_x = (int)std::floor(x0 < x1 ? x0 : x1), tmax_x = (int)std::ceil(x0 < x1 ? x1 : x0);
  const int tmin_y = (int)std::floor(y0 < y1 ? y0 : y1), tmax_y = (int)std::ceil(y0 < y1 ? y1 : y0);
  const int R0 = dcn::options().bwd_halo;
  long long best = -1;
  for (int TW = 1; TW <= 256 && TW <= g.Wo; ++TW) {
    const int TH = std::min(g.Ho, 256 / TW);
    dcn::WinGeom c;
    c.TH = TH;
    c.TW = TW;
    c.tiles_h = (g.Ho + TH - 1) / TH;
    c.tiles_w = (g.Wo + TW - 1) / TW;
    for (int R = R0; R >= 1; --R) {
      c.WH = (TH - 1) * p->stride_h + (tmax_y - tmin_y) + 2 * R + 2;
      c.WW = (TW - 1) * p->stride_w + (tmax_x - tmin_x) + 2 * R + 2;
      c.org_y = -p->pad_h + ch + tmin_y - R;
      c.org_x = -p->pad_w + cw + tmin_x - R;
      if (dcn::split_smem_bytes(c, g.P, p->gc, es) <= kSplitSmem) break;
    }
    if (dcn::split_smem_bytes(c, g.P, p->gc, es) > kSplitSmem) continue;
    const long long cost = (long long)c.tiles_h * c.tiles_w * (256 + (long long)c.WH * c.WW);
    if (best < 0 || cost < best) {
      best = cost;
      *wg = c;
    }
  }
  if (best < 0 || (long long)p->N * p->G * wg->tiles_h * wg->tiles_w > INT_MAX) return 0;
  // one input block per (image, group) plane, its window covering every
  // bilinear cell that touches the image (cells y0 in [-1, H-1], x0 in
  // [-1, W-1]): that block alone sums the plane's grad_input and writes it in
  // the storage type, with no float32 accumulator to clear and round
  wg->direct = dcn::options().bwd_direct && wg->tiles_h == 1 && wg->tiles_w == 1 &&
               wg->org_y <= -1 && wg->org_x <= -1 && wg->org_y + wg->WH - 2 >= p->H - 1 &&
               wg->org_x + wg->WW - 2 >= p->W - 1;
  // the sample blocks read their corners through L1 over the wide forward's
  // tiles (staging their windows by a tensor copy measured slower inside the
  // fused launch: FlashInternImage-T stage 1 315-326 us against 272 us, the
  // input blocks then getting less L1)
  plan_fwd_tiles(p, g, cpt, kp);
  // grad_offset / grad_mask rows staged in shared memory
  const int ub = 256 / chunks;
  if (kp->merged) {
    *la = kp->os_off;
    *lb = 0;
  } else {
    *la = 2 * g.P;
    *lb = g.P;
  }
  if (!dcn::options().bwd_stage ||
      (size_t)ub * (dcn::stage_stride(*la, es) + *lb) * es > kStageSmem)
    *la = *lb = 0;
  return cpt;
}

// The CUDA error behind this thread's last DCN_ERR_CUDA (a test hook reads it).
thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DCN_OK;
  g_last_cuda_error = (int)e;
  return DCN_ERR_CUDA;
}

// The status bits of the range checks seen by this thread's last call (the
// DCN_DEBUG_BOUNDS build; a test hook reads them).
thread_local unsigned g_last_bounds = 0;

using BoundsReader = cudaError_t (*)(unsigned*);
constexpr BoundsReader kBoundsReaders[] = {dcn::bounds_status_fwd, dcn::bounds_status_fwd_tma,
                                           dcn::bounds_status_bwd, dcn::bounds_status_bwd_split,
                                           dcn::bounds_status_dwconv, dcn::bounds_status_fwd_proj};

// The end of every call that launched work.  In the DCN_DEBUG_BOUNDS build:
// wait for the stream, collect and clear the range checks' status words, and
// report DCN_ERR_INTERNAL if any check failed; otherwise rc unchanged.
int finish(int rc, void* stream) {
#ifdef DCN_DEBUG_BOUNDS
  if (rc != DCN_OK) return rc;
  if (cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != DCN_OK)
    return DCN_ERR_CUDA;
  unsigned any = 0;
  for (BoundsReader f : kBoundsReaders) {
    unsigned v = 0;
    if (cuda_status(f(&v)) != DCN_OK) return DCN_ERR_CUDA;
    any |= v;
  }
  g_last_bounds = any;
  return any ? DCN_ERR_INTERNAL : DCN_OK;
#else
  (void)stream;
  return rc;
#endif
}

}  // namespace

extern "C" {

int dcn_out_shape(const dcn_params_t* p, int* H_out, int* W_out) {
  if (!H_out || !W_out) return DCN_ERR_NULL;
  Geometry g;
  int rc = validate(p, &g);
  if (rc != DCN_OK) return rc;
  *H_out = g.Ho;
  *W_out = g.Wo;
  return DCN_OK;
}

int dcn_num_points(const dcn_params_t* p) {
  Geometry g;
  int rc = validate(p, &g);
  return rc != DCN_OK ? -rc : g.P;
}

}  // extern "C"

namespace {

int cfs_vbytes(int gc, int es, bool bwd, std::initializer_list<const void*> ptrs);

// The output projection after the core: y (N, Ho, Wo, n_out) = out w^T + bias.
struct OutArgs {
  const void* w;
  const void* bias;
  int n_out;
  void* y;
};

// Both layouts of the offsets and masks: separate tensors (row strides 2P and
// P) or one merged tensor (offset row, then mask row, in rows of
// row_stride elements).  cfs: the centre feature scale follows, with x_proj
// the input and one logit per unit (an output the input's size, stride 1):
// in the TMA forward's epilogue for 16-bit storage, else as a second launch
// over the output in place.  oa: the output projection follows, in the TMA
// forward's epilogue where it applies (output, the core's, then unused and
// may be NULL), else as a launch of the linear kernels over output.
int core_fwd(const dcn_params_t* p, const void* input, const void* offset, const void* mask,
             void* output, void* stream, int row_stride, bool cfs = false,
             const void* logits = nullptr, const OutArgs* oa = nullptr) {
  Geometry g;
  int rc = validate(p, &g);
  if (rc != DCN_OK) return rc;
  if (row_stride && (row_stride < 3 * g.P || row_stride % 2)) return DCN_ERR_SHAPE;
  if (cfs && (p->stride_h != 1 || p->stride_w != 1 || g.Ho != p->H || g.Wo != p->W))
    return DCN_ERR_SHAPE;
  if (oa && oa->n_out < 1) return DCN_ERR_SHAPE;
  if (g.units == 0) return DCN_OK;
  if (!input || !offset || !mask || (!output && !oa) || (cfs && !logits) ||
      (oa && (!oa->w || !oa->y)))
    return DCN_ERR_NULL;
  const size_t es = (size_t)elem_size(p->dtype);
  if (!aligned(input, es) || !aligned(mask, es) || (output && !aligned(output, es)) ||
      !aligned(offset, 2 * es) || (cfs && !aligned(logits, es)) ||
      (oa && (!aligned(oa->w, es) || !aligned(oa->y, es) || (oa->bias && !aligned(oa->bias, es)))))
    return DCN_ERR_ALIGN;
  dcn::KParams kp;
  fill_kparams(p, g, &kp);
  if (row_stride) {
    kp.os_off = kp.os_mask = row_stride;
    kp.merged = 1;
    kp.merged_rows64 = g.P == 9 && es == 2 && aligned(offset, 32) &&
                       (row_stride * es) % 32 == 0 && dcn::options().fwd_row64;
  }
  const int cpt = pick_fwd_cpt(p, g, input, output);
  alignas(64) unsigned char map[128];
  dcn::TileGeom tg;
  // a window whose halo within three blocks' shared memory is under 4 pixels
  // (7 x 7 taps at stage 1: 3) takes up to two blocks' worth instead, so that
  // fewer samples leave it for the far path (FlashInternImage-T stage 1, 7 x 7:
  // 808 -> 573 us; 5 x 5, whose halo is 4, measured slower that way: 209 -> 221)
  int halo = -1;
  bool tile = cpt < 0 && plan_fwd_tile(p, g, -cpt, input, &kp, &tg, map, kTileSmem,
                                       dcn::options().fwd_any_tile != 0, &halo);
  const size_t big = (size_t)std::max(16, std::min(dcn::options().fwd_big_win, 200)) * 1024;
  if (tile && halo < 4 && halo < dcn::options().fwd_halo && big > kTileSmem)
    tile = plan_fwd_tile(p, g, -cpt, input, &kp, &tg, map, big, dcn::options().fwd_any_tile != 0);
  if (cpt < 0 && !tile) plan_fwd_tiles(p, g, -cpt, &kp);
  // the projection in the epilogue, when there is no room for the core's
  // output (with room, the two launches measure faster: the linear reads the
  // output back from L2, while the epilogue's work lengthens every block of a
  // forward that is bound by instruction issue): 16-bit, separate tensors, 64 channels in one block
  // (all groups), at most 64 tile pixels, n_out a multiple of 16 up to 128,
  // weight and y 16-byte aligned
  alignas(64) unsigned char wmap[128];
  const bool fused_out =
      oa && (dcn::options().fwd_out == 2 || (dcn::options().fwd_out == 1 && !output)) && tile &&
      es == 2 && !row_stride &&
      p->G * p->gc == 64 && tg.ngb == 1 && kp.tile_w * kp.tile_h <= 64 &&
      (-cpt == 8 || -cpt == 16) && oa->n_out % 16 == 0 &&
      oa->n_out <= 128 && aligned(oa->w, 16) && aligned(oa->y, 16) &&
      dcn::encode_out_weight_map(p->dtype, oa->w, oa->n_out, wmap);
  if (oa && !fused_out && !output) return DCN_ERR_UNSUPPORTED;  // nowhere to put the core's output
  if (fault_injected()) return DCN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool fused = cfs && tile && es == 2 && !row_stride && (dcn::options().fwd_cfs || fused_out);
  cudaError_t e =
      tile ? dcn::launch_fwd_tile(map, kp, tg, p->dtype, -cpt, input, offset, mask, output, st,
                                  fused ? logits : nullptr, fused_out ? wmap : nullptr,
                                  fused_out ? oa->bias : nullptr, fused_out ? oa->y : nullptr,
                                  fused_out ? oa->n_out : 0)
           : dcn::launch_fwd(kp, p->dtype, cpt, input, offset, mask, output, st);
  if (e == cudaSuccess && cfs && !fused) {
    const int gc = p->gc;
    e = dcn::launch_cfs_fwd(p->dtype, cfs_vbytes(gc, (int)es, false, {output, input, output}),
                            (long long)p->N * g.Ho * g.Wo, p->G * gc, p->G, output, input, logits,
                            output, st);
  }
  if (e == cudaSuccess && oa && !fused_out) {
    const long long M = (long long)p->N * g.Ho * g.Wo;
    const int C = p->G * p->gc;
    const bool tc = dcn::options().linear_tc &&
                    dcn::linear_tc_ok(p->dtype, M, C, oa->n_out, output, oa->w, oa->y);
    e = dcn::launch_linear(p->dtype, M, C, oa->n_out, output, oa->w, oa->bias, oa->y, tc, st);
  }
  return finish(cuda_status(e), stream);
}

}  // namespace

extern "C" {

int dcn_core_fwd(const dcn_params_t* p, const void* input, const void* offset, const void* mask,
                 void* output, void* stream) {
  return core_fwd(p, input, offset, mask, output, stream, 0);
}

int dcn_core_fwd_cfs(const dcn_params_t* p, const void* input, const void* offset,
                     const void* mask, const void* logits, void* output, void* stream) {
  return core_fwd(p, input, offset, mask, output, stream, 0, true, logits);
}

int dcn_core_fwd_out(const dcn_params_t* p, const void* input, const void* offset,
                     const void* mask, const void* logits, const void* weight, const void* bias,
                     int n_out, void* y, void* scratch, void* stream) {
  const OutArgs oa{weight, bias, n_out, y};
  return core_fwd(p, input, offset, mask, scratch, stream, 0, logits != nullptr, logits, &oa);
}

int dcn_core_fwd_om(const dcn_params_t* p, const void* input, const void* offset_mask,
                    int row_stride, void* output, void* stream) {
  if (row_stride <= 0) return p ? DCN_ERR_SHAPE : DCN_ERR_NULL;
  const int P = dcn_num_points(p);
  if (P < 0) return -P;
  const size_t es = (size_t)elem_size(p->dtype);
  const char* om = static_cast<const char*>(offset_mask);
  return core_fwd(p, input, om, om ? om + 2 * P * es : nullptr, output, stream, row_stride);
}

size_t dcn_core_bwd_workspace(const dcn_params_t* p) {
  Geometry g;
  if (validate(p, &g) != DCN_OK) return 0;
  return p->dtype == DCN_F32 ? 0 : (size_t)g.n_in * sizeof(float);
}

}  // extern "C"

namespace {

int core_bwd(const dcn_params_t* p, const void* grad_out, const void* input, const void* offset,
             const void* mask, void* grad_input, void* grad_offset, void* grad_mask,
             void* workspace, size_t workspace_bytes, void* stream, int row_stride) {
  Geometry g;
  int rc = validate(p, &g);
  if (rc != DCN_OK) return rc;
  if (row_stride && (row_stride < 3 * g.P || row_stride % 2)) return DCN_ERR_SHAPE;
  if (g.units == 0) return DCN_OK;
  if (!grad_out || !input || !offset || !mask || !grad_input || !grad_offset || !grad_mask)
    return DCN_ERR_NULL;
  const size_t es = (size_t)elem_size(p->dtype);
  if (!aligned(grad_out, es) || !aligned(input, es) || !aligned(mask, es) ||
      !aligned(offset, 2 * es) || !aligned(grad_input, es) || !aligned(grad_offset, es) ||
      !aligned(grad_mask, es))
    return DCN_ERR_ALIGN;
  float* acc;
  const size_t acc_bytes = (size_t)g.n_in * sizeof(float);
  if (p->dtype == DCN_F32) {
    acc = static_cast<float*>(grad_input);
  } else {
    if (!workspace || workspace_bytes < acc_bytes) return DCN_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return DCN_ERR_ALIGN;
    acc = static_cast<float*>(workspace);
  }
  dcn::KParams kp;
  fill_kparams(p, g, &kp);
  if (row_stride) {
    kp.os_off = kp.os_mask = row_stride;
    kp.merged = 1;
    kp.merged_rows64 = g.P == 9 && es == 2 && aligned(offset, 32) &&
                       (row_stride * es) % 32 == 0 && dcn::options().fwd_row64;
  }
  dcn::WinGeom wg{};
  int la = 0, lb = 0;
  const int scpt = plan_split(p, g, input, grad_out, acc, &kp, &wg, &la, &lb);
  const int cpt = scpt ? 0 : pick_bwd_cpt(p, input, grad_out, acc);
  if (fault_injected()) return DCN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g.n_in > 0 && !(scpt && wg.direct)) {
    cudaError_t e = cudaMemsetAsync(acc, 0, acc_bytes, s);
    if (e != cudaSuccess) return DCN_ERR_CUDA;
  }
  if (scpt)
    return finish(cuda_status(dcn::launch_bwd_split(kp, wg, p->dtype, scpt, la, lb, grad_out,
                                                    input, offset, mask, acc, grad_input,
                                                    grad_offset, grad_mask, s)),
                  s);
  return finish(cuda_status(dcn::launch_bwd(kp, p->dtype, cpt, grad_out, input, offset, mask,
                                            acc, grad_input, grad_offset, grad_mask, s)),
                s);
}

}  // namespace

namespace {

// The widest access (16, 8, 4 bytes or one element) that divides a group's
// bytes and to which every pointer is aligned; for the backward also with
// gc / V a power of two <= 32 (the shuffle reduction), else 0.
int cfs_vbytes(int gc, int es, bool bwd, std::initializer_list<const void*> ptrs) {
  for (int vb = 16; vb >= es; vb /= 2) {
    if ((gc * es) % vb) continue;
    bool ok = true;
    for (const void* q : ptrs) ok = ok && aligned(q, vb);
    if (!ok) continue;
    const int L = gc / (vb / es);
    if (bwd && (L > 32 || (L & (L - 1)))) continue;
    return vb;
  }
  return bwd ? 0 : es;
}

int cfs_check(const dcn_cfs_params_t* p, int* es) {
  if (!p) return DCN_ERR_NULL;
  *es = elem_size(p->dtype);
  if (*es == 0) return DCN_ERR_DTYPE;
  if (p->M < 0 || p->C < 1 || p->G < 1 || p->C % p->G) return DCN_ERR_SHAPE;
  if (p->M >= (1LL << 40) / p->C) return DCN_ERR_UNSUPPORTED;
  return DCN_OK;
}

}  // namespace

namespace {

// Shared memory the tiled feature-step kernel takes per block: within
// kDwSmemTwo two blocks fit on an SM; up to kDwSmemOne, one.
constexpr size_t kDwSmemTwo = 110 * 1024;
constexpr size_t kDwSmemOne = 220 * 1024;

// Validates a feature-step call and picks its kernel: the tiled one when the
// shape and the alignments allow, with about 128 threads a block (patches
// from C; a 512-channel patch takes 256), 4-row patches unless only 2-row
// ones let two blocks share an SM, and as many patches as then fit; else the
// one-warp-per-pixel kernel.
int dwconv_plan(const dcn_dwconv_params_t* p, const void* x, const void* w, const void* b,
                const void* g, const void* bt, const void* y, dcn::DwGeom* d) {
  if (!p) return DCN_ERR_NULL;
  const int es = elem_size(p->dtype);
  if (es == 0) return DCN_ERR_DTYPE;
  if (p->N < 0 || p->H < 1 || p->W < 1 || p->C < 1 || p->k < 1 || p->k % 2 == 0 ||
      p->k > DCN_DW_MAX_KERNEL || !(p->eps >= 0.f) || !std::isfinite(p->eps))
    return DCN_ERR_SHAPE;
  if (p->C > DCN_DW_MAX_CHANNELS) return DCN_ERR_UNSUPPORTED;
  const long long hw = (long long)p->H * p->W;
  if (p->H > kMaxExtent || p->W > kMaxExtent || (long long)p->N * hw > (1LL << 40) / p->C)
    return DCN_ERR_UNSUPPORTED;
  *d = dcn::DwGeom{p->N, p->H, p->W, p->C, p->k, p->eps, false, 1, 1, 4};
  if ((long long)p->N * hw == 0) return DCN_OK;
  if (!x || !w || !g || !bt || !y) return DCN_ERR_NULL;
  for (const void* q : {x, w, g, bt, y})
    if (!aligned(q, es)) return DCN_ERR_ALIGN;
  if (b && !aligned(b, es)) return DCN_ERR_ALIGN;
  const dcn::Options& o = dcn::options();
  bool tiled = o.dw_tiled && (p->k == 3 || p->k == 5) &&
               (p->C == 64 || p->C == 128 || p->C == 256 || p->C == 512) && aligned(x, 16);
  for (const void* q : {w, b, g, bt, y}) tiled = tiled && (!q || aligned(q, 2 * es));
  if (tiled) {
    int np0 = std::max(1, 128 / (p->C / 2));  // 128 threads measured faster than 256
    if (o.dw_patches > 0) np0 = std::min(o.dw_patches, std::max(1, 256 / (p->C / 2)));
    np0 = 1 << (31 - __builtin_clz((unsigned)np0));  // a power of two
    // 4-row patches first (fewer footprint reads per output), then 2-row;
    // each at two blocks per SM, else one (4-row patches at one block per SM
    // beat 2-row at two: InternImage-G stage 1, C = 512, 61.6 -> 59.4 us)
    for (const int py : {4, 2}) {
      if (o.dw_py && py != o.dw_py) continue;
      for (const size_t cap : {kDwSmemTwo, kDwSmemOne}) {
        for (int np = np0; np >= 1 && !d->tiled; np /= 2) {
          d->ph = np >= 4 ? 2 : 1;
          d->pw = np / d->ph;
          d->py = py;
          d->tiled = true;  // dwconv_smem_bytes sizes the tiled kernel's buffers
          d->tiled = dcn::dwconv_smem_bytes(*d, es) <= cap;
        }
        if (d->tiled) break;
      }
      if (d->tiled) break;
    }
  }
  if (!d->tiled) d->ph = d->pw = 1, d->py = 4;
  return DCN_OK;
}

}  // namespace

extern "C" {

int dcn_core_bwd(const dcn_params_t* p, const void* grad_out, const void* input,
                 const void* offset, const void* mask, void* grad_input, void* grad_offset,
                 void* grad_mask, void* workspace, size_t workspace_bytes, void* stream) {
  return core_bwd(p, grad_out, input, offset, mask, grad_input, grad_offset, grad_mask,
                  workspace, workspace_bytes, stream, 0);
}

int dcn_core_bwd_om(const dcn_params_t* p, const void* grad_out, const void* input,
                    const void* offset_mask, int row_stride, void* grad_input,
                    void* grad_offset_mask, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (row_stride <= 0) return p ? DCN_ERR_SHAPE : DCN_ERR_NULL;
  const int P = dcn_num_points(p);
  if (P < 0) return -P;
  const size_t es = (size_t)elem_size(p->dtype);
  const char* om = static_cast<const char*>(offset_mask);
  char* gom = static_cast<char*>(grad_offset_mask);
  return core_bwd(p, grad_out, input, om, om ? om + 2 * P * es : nullptr, grad_input, gom,
                  gom ? gom + 2 * P * es : nullptr, workspace, workspace_bytes, stream,
                  row_stride);
}

const char* dcn_status_str(int status) {
  switch (status) {
    case DCN_OK: return "DCN_OK";
    case DCN_ERR_NULL: return "DCN_ERR_NULL: a required pointer is NULL";
    case DCN_ERR_SHAPE: return "DCN_ERR_SHAPE: a size or geometry parameter is out of range";
    case DCN_ERR_DTYPE: return "DCN_ERR_DTYPE: unknown dtype";
    case DCN_ERR_ALIGN: return "DCN_ERR_ALIGN: a pointer is misaligned for its element type";
    case DCN_ERR_UNSUPPORTED: return "DCN_ERR_UNSUPPORTED: outside the limits of this build";
    case DCN_ERR_CUDA: return "DCN_ERR_CUDA: a CUDA call or kernel launch failed";
    case DCN_ERR_INTERNAL: return "DCN_ERR_INTERNAL: internal consistency check failed";
    case DCN_ERR_WORKSPACE: return "DCN_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown dcn status";
  }
}

int dcn_version(void) { return 100; }

int dcn_wait_timeouts(unsigned long long* count) {
  if (!count) return DCN_ERR_NULL;
  unsigned long long a = 0, c = 0, f = 0;
  if (dcn::read_wait_timeouts(&a) != cudaSuccess ||
      dcn::read_linear_wait_timeouts(&c) != cudaSuccess ||
      dcn::read_proj_wait_timeouts(&f) != cudaSuccess)
    return DCN_ERR_CUDA;
  *count = a + c + f;
  return DCN_OK;
}

int dcn_linear(const dcn_linear_params_t* p, const void* x, const void* w, const void* bias,
               void* y, void* stream) {
  if (!p) return DCN_ERR_NULL;
  const int es = elem_size(p->dtype);
  if (es == 0) return DCN_ERR_DTYPE;
  if (p->M < 0 || p->K < 1 || p->N < 1) return DCN_ERR_SHAPE;
  if (p->M > (1LL << 40) / p->K || p->M > (1LL << 40) / p->N) return DCN_ERR_UNSUPPORTED;
  if (p->M == 0) return DCN_OK;
  if (!x || !w || !y) return DCN_ERR_NULL;
  if (!aligned(x, es) || !aligned(w, es) || !aligned(y, es) || (bias && !aligned(bias, es)))
    return DCN_ERR_ALIGN;
  const bool tc = dcn::options().linear_tc && dcn::linear_tc_ok(p->dtype, p->M, p->K, p->N,
                                                                   x, w, y);
  if (fault_injected()) return DCN_ERR_CUDA;
  return finish(cuda_status(dcn::launch_linear(p->dtype, p->M, p->K, p->N, x, w, bias, y, tc,
                                        static_cast<cudaStream_t>(stream))),
                stream);
}


int dcn_center_feature_scale(const dcn_cfs_params_t* p, const void* core, const void* x_proj,
                             const void* logits, void* out, void* stream) {
  int es = 0;
  if (const int rc = cfs_check(p, &es)) return rc;
  if (p->M == 0) return DCN_OK;
  if (!core || !x_proj || !logits || !out) return DCN_ERR_NULL;
  for (const void* q : {core, x_proj, logits, (const void*)out})
    if (!aligned(q, es)) return DCN_ERR_ALIGN;
  const int vb = cfs_vbytes(p->C / p->G, es, false, {core, x_proj, out});
  if (fault_injected()) return DCN_ERR_CUDA;
  return finish(cuda_status(dcn::launch_cfs_fwd(p->dtype, vb, p->M, p->C, p->G, core, x_proj, logits,
                                         out, static_cast<cudaStream_t>(stream))),
                stream);
}

int dcn_center_feature_scale_bwd(const dcn_cfs_params_t* p, const void* grad_out,
                                 const void* core, const void* x_proj, const void* logits,
                                 void* grad_core, void* grad_x_proj, void* grad_logits,
                                 void* stream) {
  int es = 0;
  if (const int rc = cfs_check(p, &es)) return rc;
  if (p->M == 0) return DCN_OK;
  if (!grad_out || !core || !x_proj || !logits || !grad_core || !grad_x_proj || !grad_logits)
    return DCN_ERR_NULL;
  for (const void* q : {grad_out, core, x_proj, logits, (const void*)grad_core,
                        (const void*)grad_x_proj, (const void*)grad_logits})
    if (!aligned(q, es)) return DCN_ERR_ALIGN;
  const int vb = cfs_vbytes(p->C / p->G, es, true,
                            {grad_out, core, x_proj, grad_core, grad_x_proj});
  if (fault_injected()) return DCN_ERR_CUDA;
  return finish(cuda_status(dcn::launch_cfs_bwd(p->dtype, vb, p->M, p->C, p->G, grad_out, core, x_proj,
                                         logits, grad_core, grad_x_proj, grad_logits,
                                         static_cast<cudaStream_t>(stream))),
                stream);
}

int dcn_core_fwd_proj(const dcn_params_t* p, const void* input, const void* feat, int K,
                      const void* weight, const void* bias, int row_stride, void* output,
                      void* offset_mask, void* stream) {
  Geometry g;
  int rc = validate(p, &g);
  if (rc != DCN_OK) return rc;
  if (row_stride < 3 * g.P || row_stride % 2 || K < 1) return DCN_ERR_SHAPE;
  const long long nom = (long long)p->G * row_stride;
  if (g.units == 0) return DCN_OK;
  if (!input || !feat || !weight || !output) return DCN_ERR_NULL;
  const size_t es = (size_t)elem_size(p->dtype);
  for (const void* q : {input, feat, weight, (const void*)output})
    if (!aligned(q, es)) return DCN_ERR_ALIGN;
  if ((bias && !aligned(bias, es)) || (offset_mask && !aligned(offset_mask, 2 * es)))
    return DCN_ERR_ALIGN;
  const long long M = g.units / p->G;  // output pixels: the projection's rows
  if (M > (1LL << 40) / K || M > (1LL << 40) / nom || nom > INT_MAX) return DCN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // the fused launch: 16-bit storage, a tile of the TMA forward, K a multiple
  // of 64 up to 256, rows a multiple of 8 elements, 16-byte aligned tensors
  // With offset_mask given, the projection and the core as two launches are
  // faster at every measured shape (the rows then cost a trip through memory,
  // but the forward reads them with wide loads at its full occupancy); the
  // single launch serves calls without a rows buffer, which cannot allocate one.
  const dcn::Options& o = dcn::options();
  bool fused = (o.fwd_proj == 2 || (o.fwd_proj == 1 && !offset_mask)) && es == 2 &&
               K % 64 == 0 && K <= 256 && row_stride % 8 == 0 &&
               aligned(feat, 16) && aligned(weight, 16) && (!offset_mask || aligned(offset_mask, 16));
  dcn::KParams kp;
  fill_kparams(p, g, &kp);
  kp.os_off = kp.os_mask = row_stride;
  kp.merged = 1;
  alignas(64) unsigned char map[128], fmap[128], wmap[128];
  dcn::TileGeom tg;
  dcn::ProjGeom pg;
  int cpt = 0;
  if (fused) {
    cpt = pick_fwd_cpt(p, g, input, output);
    fused = cpt < 0;
    bool planned = false;
    if (fused && o.fwd_proj_ws) {
      // the persistent kernel: the tile first (its shape does not depend on
      // the budget), then the window that the other buffers leave room for
      dcn::KParams k1 = kp;
      dcn::TileGeom t1;
      if (plan_fwd_tile(p, g, -cpt, input, &k1, &t1, map, 64 * 1024, o.fwd_any_tile != 0)) {
        const size_t budget = dcn::proj_ws_window_budget(k1, t1, (int)es, K, row_stride);
        planned = budget > 0 &&
                  plan_fwd_tile(p, g, -cpt, input, &kp, &tg, map, budget, o.fwd_any_tile != 0) &&
                  dcn::proj_plan_ws(kp, tg, (int)es, K, row_stride, -cpt, &pg);
      }
    }
    if (fused && !planned)
      planned = plan_fwd_tile(p, g, -cpt, input, &kp, &tg, map,
                              (size_t)std::max(1, o.fwd_proj_win) * 1024, o.fwd_any_tile != 0) &&
                dcn::proj_plan(kp, tg, (int)es, K, row_stride, &pg);
    fused = fused && planned && dcn::encode_proj_maps(kp, pg, p->dtype, feat, K, weight, fmap, wmap);
  }
  if (fault_injected()) return DCN_ERR_CUDA;
  if (fused)
    return finish(cuda_status(dcn::launch_fwd_proj(map, fmap, wmap, kp, tg, pg, p->dtype, -cpt,
                                                   input, bias, output, offset_mask, s)),
                  stream);
  // otherwise the two launches: the projection into offset_mask, then the core
  if (!offset_mask) return DCN_ERR_UNSUPPORTED;
  const dcn_linear_params_t lp{M, K, (int)nom, p->dtype};
  rc = dcn_linear(&lp, feat, weight, bias, offset_mask, stream);
  if (rc != DCN_OK) return rc;
  return dcn_core_fwd_om(p, input, offset_mask, row_stride, output, stream);
}

int dcn_dwconv_ln_gelu(const dcn_dwconv_params_t* p, const void* x, const void* weight,
                       const void* bias, const void* gamma, const void* beta, void* y,
                       void* stream) {
  dcn::DwGeom d{};
  if (const int rc = dwconv_plan(p, x, weight, bias, gamma, beta, y, &d)) return rc;
  if ((long long)p->N * p->H * p->W == 0) return DCN_OK;
  if (fault_injected()) return DCN_ERR_CUDA;
  return finish(cuda_status(dcn::launch_dwconv(d, p->dtype, x, weight, bias, gamma, beta, y,
                                        static_cast<cudaStream_t>(stream))),
                stream);
}

}  // extern "C"

// ---- the selection switches and their test hook ----------------------------

namespace dcn {
namespace {
Options g_options;
}
const Options& options() { return g_options; }
}  // namespace dcn

namespace {
struct OptionName {
  const char* name;
  int dcn::Options::*field;
};
constexpr OptionName kOptionNames[] = {
    {"fwd_wide", &dcn::Options::fwd_wide},
    {"fwd_wide_cpt", &dcn::Options::fwd_wide_cpt},
    {"fwd_cpt", &dcn::Options::fwd_cpt},
    {"fwd_tile", &dcn::Options::fwd_tile},
    {"fwd_tma", &dcn::Options::fwd_tma},
    {"fwd_halo", &dcn::Options::fwd_halo},
    {"fwd_big_win", &dcn::Options::fwd_big_win},
    {"fwd_any_tile", &dcn::Options::fwd_any_tile},
    {"fwd_row64", &dcn::Options::fwd_row64},
    {"fwd_cfs", &dcn::Options::fwd_cfs},
    {"fwd_out", &dcn::Options::fwd_out},
    {"fwd_proj", &dcn::Options::fwd_proj},
    {"fwd_proj_win", &dcn::Options::fwd_proj_win},
    {"fwd_proj_ws", &dcn::Options::fwd_proj_ws},
    {"bwd_split", &dcn::Options::bwd_split},
    {"bwd_fuse", &dcn::Options::bwd_fuse},
    {"bwd_cpt", &dcn::Options::bwd_cpt},
    {"bwd_halo", &dcn::Options::bwd_halo},
    {"bwd_stage", &dcn::Options::bwd_stage},
    {"bwd_direct", &dcn::Options::bwd_direct},
    {"linear_tc", &dcn::Options::linear_tc},
    {"linear_bn", &dcn::Options::linear_bn},
    {"linear_yb", &dcn::Options::linear_yb},
    {"linear_s", &dcn::Options::linear_s},
    {"linear_ctas", &dcn::Options::linear_ctas},
    {"linear_persist", &dcn::Options::linear_persist},
    {"dw_tiled", &dcn::Options::dw_tiled},
    {"dw_patches", &dcn::Options::dw_patches},
    {"dw_py", &dcn::Options::dw_py},
    {"fault_inject", &dcn::Options::fault_inject},
};
}  // namespace

// Test hooks, exported but not part of the public header: set one selection
// switch by name (DCN_ERR_SHAPE for an unknown name), or put all of them back
// to their defaults.  Not for concurrent use with calls on other threads.
extern "C" int dcn_internal_set_option(const char* name, int value) {
  if (!name) return DCN_ERR_NULL;
  for (const OptionName& o : kOptionNames)
    if (std::strcmp(o.name, name) == 0) {
      dcn::g_options.*o.field = value;
      return DCN_OK;
    }
  return DCN_ERR_SHAPE;
}

extern "C" void dcn_internal_reset_options(void) { dcn::g_options = dcn::Options(); }

// Test hook: the cudaError_t behind the calling thread's last DCN_ERR_CUDA
// from a CUDA call (0 if none).
extern "C" int dcn_internal_last_cuda_error(void) { return g_last_cuda_error; }

// Test hooks of the range checks: whether this is the DCN_DEBUG_BOUNDS build;
// the status bits the calling thread's last call collected; and a status
// word set from the host (the forward's), so that the next call's check of
// the words can be seen to report DCN_ERR_INTERNAL and to clear them.
extern "C" int dcn_internal_debug_bounds(void) {
#ifdef DCN_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}
extern "C" unsigned dcn_internal_bounds_status(void) { return g_last_bounds; }
extern "C" int dcn_internal_set_bounds_status(unsigned v) {
  return cuda_status(dcn::bounds_status_set_fwd(v));
}
