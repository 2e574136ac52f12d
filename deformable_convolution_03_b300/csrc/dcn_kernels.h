// dcn_kernels.h -- launchers of the forward and backward kernels, called by
// the C ABI layer (dcn_api.cu) after it has validated every argument.
#pragma once

#include <cuda_runtime.h>

#include "dcn_common.cuh"

namespace dcn {

// cpt: channels per thread (1, 2, 4, 8, 16 or 32; a divisor of gc whose slice
// of every tensor row starts cpt*sizeof(T)-aligned) for the general kernel;
// -cpt (cpt*sizeof(T) of 16, 32 or 64 bytes, slices 32-byte aligned when 32 or
// more) selects the wide kernel.
cudaError_t launch_fwd(const KParams& kp, int dtype, int cpt, const void* in, const void* off,
                       const void* msk, void* out, cudaStream_t s);

// cpt as above with gc/cpt a power of two no larger than 32, or 0 for the
// one-thread-per-unit kernel that takes any gc.  gin_acc: the float32
// accumulator (zeroed by the caller); when it is not gin itself, a rounding
// kernel writes gin from it afterwards.
cudaError_t launch_bwd(const KParams& kp, int dtype, int cpt, const void* gout, const void* in,
                       const void* off, const void* msk, float* gin_acc, void* gin, void* goff,
                       void* gmask, cudaStream_t s);

// float32 accumulator -> 16-bit grad_input (n elements), rounding to nearest.
cudaError_t launch_round(int dtype, const float* acc, void* out, long long n, cudaStream_t s);

// The split backward (dcn_bwd_split.cu): bwd_sample_kernel (grad_offset,
// grad_mask) with cpt as the wide forward's and the tiles in kp, then
// bwd_input_kernel (grad_input) over the windows of wg, gc*sizeof(T) of 16,
// 32 or 64 bytes, P <= 16, TH*TW <= 256.  la, lb: elements per unit of the
// staged offset and mask rows (0: written straight to memory).  gin_acc
// (float32) must be cleared by the caller; when it is not gin, it is rounded
// into gin at the end.
cudaError_t launch_bwd_split(const KParams& kp, const WinGeom& wg, int dtype, int cpt, int la,
                             int lb, const void* gout, const void* in, const void* off,
                             const void* msk, float* gin_acc, void* gin, void* goff, void* gmask,
                             cudaStream_t s);

// The TMA-staged forward (dcn_fwd_tma.cu).  encode_input_map fills the
// 128-byte tensor map of the input (dims C, W, H, N; box GB*gc x WW x WH x 1;
// out-of-range elements read as zero) and returns false when the CUDA driver
// rejects it; launch_fwd_tile runs fwd_tile_kernel with cpt as the wide
// forward's (16 to 64 bytes per slice) over the tiles of kp.
bool encode_input_map(const KParams& kp, const TileGeom& tg, int dtype, const void* input,
                      void* map_out);
// With logits (16-bit storage, separate offset / mask tensors, an output the
// input's size at stride 1), the centre feature scale is applied before the
// store (the fwd_tile_kernel CFS instance); cudaErrorInvalidValue otherwise.
// With y, the output projection y = out W^T + bias runs in the epilogue
// instead of the store of out (16-bit storage, separate tensors, 64 channels in
// one block, at most 64 tile pixels, n_out a multiple of 16 up to 128; wmap
// from encode_out_weight_map);
// cudaErrorInvalidValue otherwise.
cudaError_t launch_fwd_tile(const void* map, const KParams& kp, const TileGeom& tg, int dtype,
                            int cpt, const void* in, const void* off, const void* msk, void* out,
                            cudaStream_t s, const void* logits = nullptr,
                            const void* wmap = nullptr, const void* bias = nullptr,
                            void* y = nullptr, int n_out = 0);
bool encode_out_weight_map(int dtype, const void* w, int n_out, void* map_out);
// Blocks whose bounded wait for a tensor copy ran out, since load.
cudaError_t read_wait_timeouts(unsigned long long* count);
// The CUDA driver's cuTensorMapEncodeTiled (PFN_cuTensorMapEncodeTiled_v12000,
// to be cast by the caller), or nullptr if the CUDA driver does not provide it.
void* tensor_map_encoder();

// The forward with the merged offset/mask projection in its prologue
// (dcn_fwd_proj.cu), on a tile planned for the TMA forward: proj_plan fills
// pg (false when the shape does not fit: 16-bit only, K a multiple of 64 up to
// 256, NB a multiple of 16 up to 256, at most 128 tile pixels);
// encode_proj_maps the tensor maps of the features (K, Wo, Ho, N) and of the
// weight (K, G * row_stride); launch_fwd_proj runs it (bias may be null; om,
// the merged rows written out, may be null).
bool proj_plan(const KParams& kp, const TileGeom& tg, int es, int K, int rs, ProjGeom* pg);
// The persistent, warp-specialised version: proj_ws_window_budget gives the
// window budget its other buffers leave (0: none); proj_plan_ws fills pg
// (pg->ws = 1) for a tile planned with that budget, false if it does not fit.
size_t proj_ws_window_budget(const KParams& kp, const TileGeom& tg, int es, int K, int rs);
bool proj_plan_ws(const KParams& kp, const TileGeom& tg, int es, int K, int rs, int cpt,
                  ProjGeom* pg);
bool encode_proj_maps(const KParams& kp, const ProjGeom& pg, int dtype, const void* feat, int K,
                      const void* w, void* fmap_out, void* wmap_out);
cudaError_t launch_fwd_proj(const void* map, const void* fmap, const void* wmap,
                            const KParams& kp, const TileGeom& tg, const ProjGeom& pg, int dtype,
                            int cpt, const void* in, const void* bias, void* out, void* om,
                            cudaStream_t s);
cudaError_t read_proj_wait_timeouts(unsigned long long* count);

// The linear projections (dcn_linear.cu): the tensor-core kernels when tc
// (the shape and alignment checks of linear_tc_ok pass), else shared-memory
// tiles on the CUDA cores.
bool linear_tc_ok(int dtype, long long M, int K, int N, const void* x, const void* w,
                  const void* y);
cudaError_t launch_linear(int dtype, long long M, int K, int N, const void* x, const void* w,
                          const void* b, void* y, bool tc, cudaStream_t s);
cudaError_t read_linear_wait_timeouts(unsigned long long* count);

// The centre feature scale (dcn_cfs.cu).  vbytes: the bytes a thread moves per
// access (16, 8, 4 or the element size), dividing gc * es, with every pointer
// aligned to it.  For the backward, gc / (vbytes / es) must be a power of two
// <= 32; vbytes == 0 selects the per-(pixel, group) kernel for any gc.
cudaError_t launch_cfs_fwd(int dtype, int vbytes, long long M, int C, int G, const void* core,
                           const void* x, const void* logits, void* out, cudaStream_t s);
cudaError_t launch_cfs_bwd(int dtype, int vbytes, long long M, int C, int G, const void* gout,
                           const void* core, const void* x, const void* logits, void* gcore,
                           void* gx, void* glogits, cudaStream_t s);

// The offset branch's feature step (dcn_dwconv.cu).  tiled: the tiled kernel
// (k of 3 or 5, C of 64, 128, 256 or 512, the input 16-byte aligned and
// every other tensor aligned to two elements) with ph x pw patches of py x 4
// pixels per block (py of 2 or 4; ph * pw * C / 2 threads, at most 256);
// otherwise the one-warp-per-pixel kernel (C up to 2048).
struct DwGeom {
  int N, H, W, C, k;
  float eps;
  bool tiled;
  int ph, pw, py;
};
size_t dwconv_smem_bytes(const DwGeom& d, int es);
cudaError_t launch_dwconv(const DwGeom& d, int dtype, const void* x, const void* w, const void* b,
                          const void* g, const void* bt, void* y, cudaStream_t s);

// The range checks' status word of each translation unit that has checks
// (always 0 outside the DCN_DEBUG_BOUNDS build): read and clear; set.
cudaError_t bounds_status_fwd(unsigned* v);
cudaError_t bounds_status_fwd_tma(unsigned* v);
cudaError_t bounds_status_bwd(unsigned* v);
cudaError_t bounds_status_bwd_split(unsigned* v);
cudaError_t bounds_status_dwconv(unsigned* v);
cudaError_t bounds_status_fwd_proj(unsigned* v);
cudaError_t bounds_status_set_fwd(unsigned v);

}  // namespace dcn
