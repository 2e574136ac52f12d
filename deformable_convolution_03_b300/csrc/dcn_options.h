// dcn_options.h -- the library's kernel-selection switches.
//
// Every field holds the production default.  The library never reads the
// environment: the tests change a switch through dcn_internal_set_option (an
// exported function that the public header does not declare) to run every
// kernel instance and path against the oracle, and put it back afterwards.
#pragma once

namespace dcn {

struct Options {
  // forward
  int fwd_wide = 1;       // 0: the general kernel instead of the wide one
  int fwd_wide_cpt = 16;  // largest slice (channels) of the wide kernel
  int fwd_cpt = 0;        // largest slice of the general kernel (0: one 16-byte vector)
  int fwd_tile = 1;       // 2-D pixel tiles for the wide kernel
  int fwd_tma = 1;        // the TMA-staged forward
  int fwd_halo = 6;       // largest halo of the TMA forward's window
  int fwd_big_win = 112;  // window budget (KB) of the TMA forward when 64 KB leaves a halo under 4 (two blocks per SM)
  int fwd_any_tile = 1;   // tiles of any shape (else powers of two) for the TMA forward
  int fwd_row64 = 1;      // 256-bit loads of merged 64-byte offset/mask rows
  int fwd_cfs = 1;        // the centre feature scale in the TMA forward's epilogue (else a second launch)
  int fwd_out = 1;        // the output projection in the TMA forward's epilogue: 1 without scratch, 2 always, 0 never
  int fwd_proj = 1;       // the projection inside the forward: 1 without a rows buffer, 2 always, 0 never
  int fwd_proj_win = 40;  // window budget (KB) of the per-tile fused forward (40 measured fastest)
  int fwd_proj_ws = 1;    // the persistent, warp-specialised fused forward where it fits
  // backward
  int bwd_split = 2;      // 2: split kernels for 16-bit storage, 1: for any dtype, 0: never
  int bwd_fuse = 1;       // both split halves in one launch
  int bwd_cpt = 4;        // largest slice of the single-pass kernel
  int bwd_halo = 5;       // halo (pixels) of the split input blocks' windows (5 measured fastest)
  int bwd_stage = 1;      // gradient rows staged in shared memory
  int bwd_direct = 1;     // planes one input block covers: grad_input written directly
  // projections
  int linear_tc = 1;       // tensor-core kernels where they apply
  int linear_bn = 256;     // largest output tile width of the K-loop kernel
  int linear_yb = 2;       // its output staging buffers
  int linear_s = 8;        // its largest stage count
  int linear_ctas = 2;     // persistent CTAs per SM when they fit
  int linear_persist = 1;  // the persistent kernel where it applies
  // the offset branch's feature step
  int dw_tiled = 1;      // the tiled kernel where it applies
  int dw_patches = 0;    // patches of a tiled block, at most 256 threads (0: about 128 threads)
  int dw_py = 0;         // patch rows of the tiled kernel (2 or 4; 0: from the shared memory)
  // a valid call reports DCN_ERR_CUDA before any CUDA call (error-path tests)
  int fault_inject = 0;
};

// The switches in force (process-wide).
const Options& options();

}  // namespace dcn
